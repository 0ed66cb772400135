"""Python binding of libtwell.so, the GB300 (sm_103a) activation-sparse gated
FFN library with the TwELL format.

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  torch supplies device memory and streams.  The
functions keep the C entry points' names (see ``include/twell.h``); they take
torch tensors, pass their device pointers, and raise ``TwellError`` when the
C call returns an error.  There is no fallback: if ``libtwell.so`` has not
been built, every call raises.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

import torch

__all__ = [
    "TwellError", "TwELL", "Hybrid", "lib", "twell_gate_pack", "twell_ffn_fwd", "twell_ffn_decode",
    "twell_ffn_fwd_tc", "twell_ffn_fwd_tc_sorted", "twell_to_f16",
    "twell_to_hybrid", "twell_workspace_size", "hybrid_ffn_fwd", "hybrid_ffn_fwd_noalloc",
    "hybrid_ffn_bwd", "hybrid_ffn_fwd_tc", "hybrid_ffn_bwd_tc",
    "twell_status_string", "twell_probe_fma", "twell_gate_pack_wait_limit",
    "FLAG_SPILL_FULL", "FLAG_DENSE_FULL", "FLAG_TIMEOUT", "FLAG_RANGE", "FLAG_BOUNDS", "TILE",
    "library",
    "WS_HYBRID_FWD", "WS_HYBRID_BWD", "WS_HYBRID_FWD_TC", "WS_HYBRID_BWD_TC", "WS_FFN_FWD_TC",
    "WS_FFN_FWD_TC_SORTED",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtwell.so")
BOUNDS_LIB_PATH = os.path.join(HERE, "libtwell_bounds.so")
TILE = 128
FLAG_SPILL_FULL = 1
FLAG_DENSE_FULL = 2
FLAG_TIMEOUT = 4
FLAG_RANGE = 8
FLAG_BOUNDS = 16

c_i32 = ctypes.c_int32
c_ptr = ctypes.c_void_p


class TwellStruct(ctypes.Structure):
    """Mirror of ``twell_t``."""
    _fields_ = [
        ("T", c_i32), ("F", c_i32), ("tile", c_i32), ("width", c_i32),
        ("val", c_ptr), ("col", c_ptr), ("cnt", c_ptr), ("spill_slot", c_ptr),
        ("spill_cap", c_i32), ("spill_n", c_ptr), ("spill_rt", c_ptr), ("spill_val", c_ptr),
        ("block_bits", c_ptr),
    ]


class HybridStruct(ctypes.Structure):
    """Mirror of ``hybrid_t``."""
    _fields_ = [
        ("T", c_i32), ("F", c_i32), ("tile", c_i32), ("cap", c_i32), ("max_dense", c_i32),
        ("n_ell", c_ptr), ("n_dense", c_ptr), ("row_map", c_ptr), ("ell_rows", c_ptr),
        ("ell_val", c_ptr), ("ell_col", c_ptr), ("ell_cnt", c_ptr), ("dense_rows", c_ptr),
        ("dense_h", c_ptr),
    ]


class TwellError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {twell_status_string(code)}")


_LIB = None

# name -> (restype, argtypes)
_SIGNATURES = {
    "twell_gate_pack": (c_i32, [c_ptr, c_ptr, c_i32, c_i32, c_i32, ctypes.POINTER(TwellStruct),
                                c_ptr, c_ptr, c_ptr]),
    "twell_ffn_fwd": (c_i32, [c_ptr, ctypes.POINTER(TwellStruct), c_ptr, c_ptr, c_i32, c_ptr,
                              c_ptr, c_ptr]),
    "twell_ffn_decode": (c_i32, [c_ptr, c_ptr, c_ptr, c_ptr, c_i32, c_i32, c_i32,
                                 ctypes.POINTER(TwellStruct), c_ptr, c_ptr, c_ptr, c_ptr]),
    "twell_ffn_fwd_tc": (c_i32, [c_ptr, ctypes.POINTER(TwellStruct), c_ptr, c_ptr, c_ptr, c_i32,
                                 c_ptr, c_ptr, ctypes.c_size_t, c_ptr, c_ptr]),
    "twell_ffn_fwd_tc_sorted": (c_i32, [c_ptr, ctypes.POINTER(TwellStruct), c_ptr, c_ptr, c_ptr,
                                        c_i32, c_ptr, c_ptr, ctypes.c_size_t, c_ptr, c_ptr]),
    "twell_to_f16": (c_i32, [c_ptr, c_ptr, ctypes.c_size_t, c_ptr, c_ptr]),
    "twell_to_hybrid": (c_i32, [ctypes.POINTER(TwellStruct), ctypes.POINTER(HybridStruct),
                                c_ptr, c_ptr]),
    "twell_workspace_size": (ctypes.c_size_t, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
    "hybrid_ffn_fwd": (c_i32, [c_ptr, ctypes.POINTER(HybridStruct), c_ptr, c_ptr, c_i32, c_ptr,
                               c_ptr, c_ptr, c_ptr, ctypes.c_size_t, c_ptr, c_ptr]),
    "hybrid_ffn_bwd": (c_i32, [c_ptr, ctypes.POINTER(HybridStruct), c_ptr, c_ptr, c_ptr, c_ptr,
                               c_ptr, c_i32, c_ptr, ctypes.c_float, c_ptr, c_ptr, c_ptr, c_ptr,
                               c_ptr, ctypes.c_size_t, c_ptr, c_ptr]),
    "hybrid_ffn_fwd_tc": (c_i32, [c_ptr, ctypes.POINTER(HybridStruct), c_ptr, c_ptr, c_i32,
                                  c_ptr, c_ptr, c_ptr, c_ptr, ctypes.c_size_t, c_ptr, c_ptr]),
    "hybrid_ffn_bwd_tc": (c_i32, [c_ptr, ctypes.POINTER(HybridStruct), c_ptr, c_ptr, c_ptr,
                                  c_ptr, c_ptr, c_i32, c_ptr, ctypes.c_float, c_ptr, c_ptr, c_ptr,
                                  c_ptr, c_ptr, ctypes.c_size_t, c_ptr, c_ptr]),
    "hybrid_ffn_fwd_noalloc": (c_i32, [c_ptr, ctypes.POINTER(HybridStruct), c_ptr, c_ptr, c_i32,
                                       c_ptr, c_ptr, c_ptr, c_ptr, c_ptr]),
    "twell_status_string": (ctypes.c_char_p, [c_i32]),
    "twell_gate_pack_wait_limit": (ctypes.c_uint64, [ctypes.c_uint64]),
    "twell_probe_fma": (c_i32, [c_i32, c_i32, c_ptr, ctypes.c_size_t,
                                ctypes.POINTER(ctypes.c_int64), c_ptr]),
    "twell_version": (c_i32, []),
}


def _load(path):
    handle = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib():
    """The loaded ``libtwell.so`` (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m activation_sparse_gated_gate_gb300.build`")
        _LIB = _load(LIB_PATH)
    return _LIB


@contextlib.contextmanager
def library(path):
    """Route this binding's calls through another build of the library at
    ``path`` (e.g. ``BOUNDS_LIB_PATH``, the bounds-checking build) inside
    the ``with`` block."""
    global _LIB
    prev = lib()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m activation_sparse_gated_gate_gb300.build`")
    _LIB = _load(path)
    try:
        yield _LIB
    finally:
        _LIB = prev


def twell_status_string(code: int) -> str:
    return lib().twell_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code, where):
    if code != 0:
        raise TwellError(code, where)


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class TwELL:
    """Device buffers of a TwELL gate activation and the ``twell_t``
    descriptor that points at them (layouts in ``include/twell.h``).

    ``spill_cap`` defaults to T * n_t slices, enough for every (row, tile)
    to overflow.  ``status`` is a device int32 the kernels OR flags into.
    ``block_bits`` (default on) adds the per-block union bitmap that the
    gate kernel fills and the tensor-core forward reads.
    """

    def __init__(self, T: int, F: int, width: int, spill_cap: int | None = None,
                 device=None, tile: int = TILE, block_bits: bool = True):
        device = torch.device(device if device is not None else "cuda")
        n_t = F // tile
        if spill_cap is None:
            spill_cap = T * n_t if width < tile else 0
        self.T, self.F, self.width, self.tile, self.n_t = T, F, width, tile, n_t
        self.spill_cap = spill_cap
        self.device = device
        self.val = torch.empty((T, n_t, width), dtype=torch.float32, device=device)
        self.col = torch.empty((T, n_t, width), dtype=torch.uint8, device=device)
        self.cnt = torch.empty((T, n_t), dtype=torch.uint8, device=device)
        self.spill_slot = torch.empty((T, n_t), dtype=torch.int32, device=device)
        self.spill_n = torch.zeros((1,), dtype=torch.int32, device=device)
        self.spill_rt = torch.empty((max(spill_cap, 1),), dtype=torch.int32, device=device)
        self.spill_val = torch.empty((max(spill_cap, 1), tile), dtype=torch.float32,
                                     device=device)
        self.status = torch.zeros((1,), dtype=torch.int32, device=device)
        self.block_bits = (torch.zeros(((T + 127) // 128, F // 32), dtype=torch.int32,
                                       device=device) if block_bits else None)
        self.struct = TwellStruct(
            T, F, tile, width, self.val.data_ptr(), self.col.data_ptr(), self.cnt.data_ptr(),
            self.spill_slot.data_ptr(), spill_cap, self.spill_n.data_ptr(),
            self.spill_rt.data_ptr(), self.spill_val.data_ptr(),
            self.block_bits.data_ptr() if block_bits else None)


def twell_gate_pack(x, Wg_t, out: TwELL, z_debug=None, status=None, stream=None):
    """Gate GEMM z = x W_g with the TwELL-packing epilogue into ``out``.
    ``z_debug`` (optional [T][F] fp32) receives z."""
    _need(x, torch.bfloat16, "x")
    _need(Wg_t, torch.bfloat16, "Wg_t")
    if z_debug is not None:
        _need(z_debug, torch.float32, "z_debug")
    status = out.status if status is None else status
    T, D = x.shape
    F = Wg_t.shape[0]
    if Wg_t.shape[1] != D:
        raise ValueError("Wg_t must be [F][D]")
    with torch.cuda.device(x.device):
        _check(lib().twell_gate_pack(_ptr(x), _ptr(Wg_t), T, D, F, ctypes.byref(out.struct),
                                     _ptr(z_debug), _ptr(status), _stream(stream)),
               "twell_gate_pack")
    return out


def twell_ffn_decode(x, Wg_t, Wu_t, Wd, out: TwELL, y=None, z_debug=None, status=None,
                     stream=None):
    """Decode-sized forward in one call (1 <= T <= 256): the gate with its
    TwELL epilogue into ``out`` (as ``twell_gate_pack``) and the up + down
    projection into y -- inside the gate kernel up to 8 tokens, else by the
    CUDA-core fused kernel after a gate kernel that prefetched the active
    rows; returns y [T][D] fp32 (allocated if not given, zeroed by the call)."""
    for t, name in ((x, "x"), (Wg_t, "Wg_t"), (Wu_t, "Wu_t"), (Wd, "Wd")):
        _need(t, torch.bfloat16, name)
    T, D = x.shape
    F = Wg_t.shape[0]
    if Wg_t.shape[1] != D or Wu_t.shape != (F, D) or Wd.shape != (F, D):
        raise ValueError("shape mismatch: x [T][D], Wg_t, Wu_t and Wd [F][D]")
    if y is None:
        y = torch.empty((T, D), dtype=torch.float32, device=x.device)
    _need(y, torch.float32, "y")
    if z_debug is not None:
        _need(z_debug, torch.float32, "z_debug")
    status = out.status if status is None else status
    with torch.cuda.device(x.device):
        _check(lib().twell_ffn_decode(_ptr(x), _ptr(Wg_t), _ptr(Wu_t), _ptr(Wd), T, D, F,
                                      ctypes.byref(out.struct), _ptr(y), _ptr(z_debug),
                                      _ptr(status), _stream(stream)),
               "twell_ffn_decode")
    return y


def twell_gate_pack_wait_limit(ns: int) -> int:
    """Set the bound (ns) on the gate kernel's pipeline waits for later
    ``twell_gate_pack`` calls (0 = the 1 s default); returns the previous."""
    return int(lib().twell_gate_pack_wait_limit(int(ns)))


def twell_ffn_fwd(x, h: TwELL, Wu_t, Wd, y=None, status=None, stream=None):
    """Fused up + down projection from the TwELL gate ``h``; returns y
    [T][D] fp32 (allocated if not given)."""
    _need(x, torch.bfloat16, "x")
    _need(Wu_t, torch.bfloat16, "Wu_t")
    _need(Wd, torch.bfloat16, "Wd")
    T, D = x.shape
    if y is None:
        y = torch.empty((T, D), dtype=torch.float32, device=x.device)
    _need(y, torch.float32, "y")
    if Wu_t.shape != (h.F, D) or Wd.shape != (h.F, D) or T != h.T:
        raise ValueError("shape mismatch: x [T][D], Wu_t and Wd [F][D]")
    status = h.status if status is None else status
    with torch.cuda.device(x.device):
        _check(lib().twell_ffn_fwd(_ptr(x), ctypes.byref(h.struct), _ptr(Wu_t), _ptr(Wd), D,
                                   _ptr(y), _ptr(status), _stream(stream)),
               "twell_ffn_fwd")
    return y


def twell_to_f16(src, dst=None, status=None, stream=None):
    """fp16 copy of a bf16 tensor (e.g. W_d for ``twell_ffn_fwd_tc``)."""
    _need(src, torch.bfloat16, "src")
    if dst is None:
        dst = torch.empty(src.shape, dtype=torch.float16, device=src.device)
    if dst.dtype != torch.float16 or not dst.is_contiguous() or dst.shape != src.shape:
        raise ValueError("dst must be a contiguous fp16 tensor shaped like src")
    if status is None:
        status = torch.zeros((1,), dtype=torch.int32, device=src.device)
    with torch.cuda.device(src.device):
        _check(lib().twell_to_f16(_ptr(src), _ptr(dst), src.numel(), _ptr(status),
                                  _stream(stream)), "twell_to_f16")
    return dst


def twell_ffn_fwd_tc(x, h: TwELL, Wu_t, Wd, y=None, ws=None, Wd_f16=None, status=None,
                     stream=None, sorted_rows=False):
    """Tensor-core (union-gather) up + down projection from the TwELL gate
    ``h``: the same function as ``twell_ffn_fwd`` with h*u rounded to fp16;
    returns y [T][D] fp32 (allocated if not given).  ``ws`` is the device
    workspace (allocated if not given); ``Wd_f16`` an optional fp16 copy of
    ``Wd`` (``twell_to_f16``), made by the call when not given.  With
    ``sorted_rows`` the call is ``twell_ffn_fwd_tc_sorted`` (token blocks
    grouped by activity)."""
    _need(x, torch.bfloat16, "x")
    _need(Wu_t, torch.bfloat16, "Wu_t")
    _need(Wd, torch.bfloat16, "Wd")
    T, D = x.shape
    if y is None:
        y = torch.empty((T, D), dtype=torch.float32, device=x.device)
    _need(y, torch.float32, "y")
    if Wu_t.shape != (h.F, D) or Wd.shape != (h.F, D) or T != h.T:
        raise ValueError("shape mismatch: x [T][D], Wu_t and Wd [F][D]")
    if Wd_f16 is not None and (Wd_f16.dtype != torch.float16 or Wd_f16.shape != Wd.shape
                               or not Wd_f16.is_contiguous()):
        raise ValueError("Wd_f16 must be a contiguous fp16 copy of Wd")
    op = WS_FFN_FWD_TC_SORTED if sorted_rows else WS_FFN_FWD_TC
    name = "twell_ffn_fwd_tc_sorted" if sorted_rows else "twell_ffn_fwd_tc"
    nbytes = twell_workspace_size(op, T, D, h.F, 0, 0)
    if ws is None:
        ws = _workspace(nbytes, x.device)
    status = h.status if status is None else status
    with torch.cuda.device(x.device):
        _check(getattr(lib(), name)(_ptr(x), ctypes.byref(h.struct), _ptr(Wu_t), _ptr(Wd),
                                    _ptr(Wd_f16), D, _ptr(y), _ptr(ws),
                                    ws.numel() * ws.element_size(), _ptr(status),
                                    _stream(stream)),
               name)
    return y


def twell_ffn_fwd_tc_sorted(x, h: TwELL, Wu_t, Wd, y=None, ws=None, Wd_f16=None, status=None,
                            stream=None):
    """``twell_ffn_fwd_tc`` on token blocks grouped by activity (rows sorted
    by their count of active neurons); same result, less GEMM work when the
    per-token activity varies widely."""
    return twell_ffn_fwd_tc(x, h, Wu_t, Wd, y=y, ws=ws, Wd_f16=Wd_f16, status=status,
                            stream=stream, sorted_rows=True)


class Hybrid:
    """Device buffers of the hybrid training format (ELL rows + dense
    backup) and the ``hybrid_t`` descriptor pointing at them."""

    def __init__(self, T: int, F: int, cap: int, max_dense: int, device=None,
                 tile: int = TILE):
        device = torch.device(device if device is not None else "cuda")
        n_t = F // tile
        self.T, self.F, self.cap, self.max_dense, self.tile, self.n_t = (
            T, F, cap, max_dense, tile, n_t)
        self.device = device
        i32 = torch.int32
        self.counts = torch.zeros((2,), dtype=i32, device=device)  # n_ell, n_dense
        self.row_map = torch.empty((max(T, 1),), dtype=i32, device=device)
        self.ell_rows = torch.empty((max(T, 1),), dtype=i32, device=device)
        self.ell_val = torch.empty((T, n_t, cap), dtype=torch.float32, device=device)
        self.ell_col = torch.empty((T, n_t, cap), dtype=torch.uint8, device=device)
        self.ell_cnt = torch.empty((T, n_t), dtype=torch.uint8, device=device)
        self.dense_rows = torch.empty((max(max_dense, 1),), dtype=i32, device=device)
        self.dense_h = torch.empty((max(max_dense, 1), F), dtype=torch.float32, device=device)
        self.status = torch.zeros((1,), dtype=i32, device=device)
        base = self.counts.data_ptr()
        self.struct = HybridStruct(
            T, F, tile, cap, max_dense, base, base + 4, self.row_map.data_ptr(),
            self.ell_rows.data_ptr(), self.ell_val.data_ptr(), self.ell_col.data_ptr(),
            self.ell_cnt.data_ptr(), self.dense_rows.data_ptr(), self.dense_h.data_ptr())

    @property
    def n_ell(self) -> int:
        return int(self.counts[0].item())

    @property
    def n_dense(self) -> int:
        return int(self.counts[1].item())


def twell_to_hybrid(h: TwELL, out: Hybrid, status=None, stream=None):
    """TwELL -> hybrid (ELL rows with capacity out.cap, dense backup)."""
    if out.T != h.T or out.F != h.F:
        raise ValueError("hybrid and TwELL shapes differ")
    status = out.status if status is None else status
    with torch.cuda.device(out.device):
        _check(lib().twell_to_hybrid(ctypes.byref(h.struct), ctypes.byref(out.struct),
                                     _ptr(status), _stream(stream)), "twell_to_hybrid")
    return out


WS_HYBRID_FWD = 1
WS_HYBRID_BWD = 2
WS_HYBRID_FWD_TC = 3
WS_HYBRID_BWD_TC = 4
WS_FFN_FWD_TC = 5
WS_FFN_FWD_TC_SORTED = 6


def twell_workspace_size(op: int, T: int, D: int, F: int, cap: int, max_dense: int) -> int:
    return int(lib().twell_workspace_size(op, T, D, F, cap, max_dense))


def _workspace(nbytes, device):
    # 256-byte aligned scratch from torch's allocator (its blocks are 512-aligned)
    return torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=device)


def hybrid_ffn_fwd(x, h: Hybrid, Wu_t, Wd, y=None, u_ell=None, U_dense=None, ws=None,
                   status=None, stream=None):
    """Hybrid training forward; returns (y, u_ell, U_dense)."""
    return _hybrid_fwd("hybrid_ffn_fwd", WS_HYBRID_FWD, x, h, Wu_t, Wd, y, u_ell, U_dense, ws,
                       status, stream)


def hybrid_ffn_fwd_tc(x, h: Hybrid, Wu_t, Wd, y=None, u_ell=None, U_dense=None, ws=None,
                      status=None, stream=None):
    """Hybrid training forward, ELL rows on the tensor cores; returns
    (y, u_ell, U_dense)."""
    return _hybrid_fwd("hybrid_ffn_fwd_tc", WS_HYBRID_FWD_TC, x, h, Wu_t, Wd, y, u_ell, U_dense,
                       ws, status, stream)


def _hybrid_fwd(name, op, x, h, Wu_t, Wd, y, u_ell, U_dense, ws, status, stream):
    _need(x, torch.bfloat16, "x")
    _need(Wu_t, torch.bfloat16, "Wu_t")
    _need(Wd, torch.bfloat16, "Wd")
    T, D = x.shape
    dev = x.device
    if y is None:
        y = torch.empty((T, D), dtype=torch.float32, device=dev)
    if u_ell is None:
        u_ell = torch.empty((T, h.n_t, h.cap), dtype=torch.float32, device=dev)
    if U_dense is None:
        U_dense = torch.empty((max(h.max_dense, 1), h.F), dtype=torch.float32, device=dev)
    need = twell_workspace_size(op, T, D, h.F, h.cap, h.max_dense)
    if ws is None:
        ws = _workspace(need, dev)
    status = h.status if status is None else status
    with torch.cuda.device(dev):
        _check(getattr(lib(), name)(_ptr(x), ctypes.byref(h.struct), _ptr(Wu_t), _ptr(Wd), D,
                                    _ptr(y), _ptr(u_ell), _ptr(U_dense), _ptr(ws),
                                    ws.numel(), _ptr(status), _stream(stream)),
               name)
    return y, u_ell, U_dense


def hybrid_ffn_bwd(x, h: Hybrid, u_ell, U_dense, Wg_t, Wu_t, Wd, dy, l1_coeff, dx=None,
                   dWg_t=None, dWu_t=None, dWd=None, ws=None, status=None, stream=None):
    """Hybrid training backward with the L1 term; returns (dx, dWg_t, dWu_t, dWd)."""
    return _hybrid_bwd("hybrid_ffn_bwd", WS_HYBRID_BWD, x, h, u_ell, U_dense, Wg_t, Wu_t, Wd, dy,
                       l1_coeff, dx, dWg_t, dWu_t, dWd, ws, status, stream)


def hybrid_ffn_bwd_tc(x, h: Hybrid, u_ell, U_dense, Wg_t, Wu_t, Wd, dy, l1_coeff, dx=None,
                      dWg_t=None, dWu_t=None, dWd=None, ws=None, status=None, stream=None):
    """Hybrid training backward, ELL rows on the tensor cores; returns
    (dx, dWg_t, dWu_t, dWd)."""
    return _hybrid_bwd("hybrid_ffn_bwd_tc", WS_HYBRID_BWD_TC, x, h, u_ell, U_dense, Wg_t, Wu_t,
                       Wd, dy, l1_coeff, dx, dWg_t, dWu_t, dWd, ws, status, stream)


def _hybrid_bwd(name, op, x, h, u_ell, U_dense, Wg_t, Wu_t, Wd, dy, l1_coeff, dx, dWg_t, dWu_t,
                dWd, ws, status, stream):
    for t, n in ((x, "x"), (Wg_t, "Wg_t"), (Wu_t, "Wu_t"), (Wd, "Wd")):
        _need(t, torch.bfloat16, n)
    _need(dy, torch.float32, "dy")
    T, D = x.shape
    F = h.F
    dev = x.device
    f32 = torch.float32
    dx = torch.empty((T, D), dtype=f32, device=dev) if dx is None else dx
    dWg_t = torch.empty((F, D), dtype=f32, device=dev) if dWg_t is None else dWg_t
    dWu_t = torch.empty((F, D), dtype=f32, device=dev) if dWu_t is None else dWu_t
    dWd = torch.empty((F, D), dtype=f32, device=dev) if dWd is None else dWd
    need = twell_workspace_size(op, T, D, F, h.cap, h.max_dense)
    if ws is None:
        ws = _workspace(need, dev)
    status = h.status if status is None else status
    with torch.cuda.device(dev):
        _check(getattr(lib(), name)(_ptr(x), ctypes.byref(h.struct), _ptr(u_ell), _ptr(U_dense),
                                    _ptr(Wg_t), _ptr(Wu_t), _ptr(Wd), D, _ptr(dy),
                                    float(l1_coeff), _ptr(dx), _ptr(dWg_t), _ptr(dWu_t),
                                    _ptr(dWd), _ptr(ws), ws.numel(), _ptr(status),
                                    _stream(stream)),
               name)
    return dx, dWg_t, dWu_t, dWd


def hybrid_ffn_fwd_noalloc(x, h: Hybrid, Wu_t, Wd, y=None, u_ell=None, U_dense=None,
                           status=None, stream=None):
    """hybrid_ffn_fwd with the library's own 64 MiB device scratch array as
    workspace (for callers that cannot allocate device memory); returns
    (y, u_ell, U_dense).  Outputs are still the caller's."""
    _need(x, torch.bfloat16, "x")
    _need(Wu_t, torch.bfloat16, "Wu_t")
    _need(Wd, torch.bfloat16, "Wd")
    T, D = x.shape
    dev = x.device
    if y is None:
        y = torch.empty((T, D), dtype=torch.float32, device=dev)
    if u_ell is None:
        u_ell = torch.empty((T, h.n_t, h.cap), dtype=torch.float32, device=dev)
    if U_dense is None:
        U_dense = torch.empty((max(h.max_dense, 1), h.F), dtype=torch.float32, device=dev)
    status = h.status if status is None else status
    with torch.cuda.device(dev):
        _check(lib().hybrid_ffn_fwd_noalloc(_ptr(x), ctypes.byref(h.struct), _ptr(Wu_t),
                                            _ptr(Wd), D, _ptr(y), _ptr(u_ell), _ptr(U_dense),
                                            _ptr(status), _stream(stream)),
               "hybrid_ffn_fwd_noalloc")
    return y, u_ell, U_dense


def twell_probe_fma(packed: bool, iters: int, out=None, stream=None, device=None):
    """Launch the FP32 FMA throughput probe (scalar or packed f32x2 chains);
    returns (out, flops) where flops = 2 * 16 * iters * threads.  The caller
    times the launch on ``stream``."""
    device = torch.device(device if device is not None else "cuda")
    n_sm = torch.cuda.get_device_properties(device).multi_processor_count
    if out is None:
        out = torch.empty((2 * n_sm * 512,), dtype=torch.float32, device=device)
    threads = ctypes.c_int64(0)
    with torch.cuda.device(device):
        _check(lib().twell_probe_fma(1 if packed else 0, int(iters), _ptr(out), out.numel(),
                                     ctypes.byref(threads), _stream(stream)),
               "twell_probe_fma")
    return out, 2.0 * 16 * iters * threads.value
