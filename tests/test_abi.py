"""The C-ABI library loads, exports every entry point include/twell.h
declares, its structs match the binding's layout, and host-side argument
validation rejects bad calls before touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import activation_sparse_gated_gate_gb300 as tw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "twell.h")

INVALID, UNSUPPORTED, CUDA = 1, 2, 3


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(\w+)\s*\([^;{]*\)\s*;", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(tw.LIB_PATH):
        from activation_sparse_gated_gate_gb300 import build
        build.build()
    return tw.lib()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "twell_gate_pack" in names and "twell_ffn_fwd" in names
    out = subprocess.run(["nm", "-D", "--defined-only", tw.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)


def test_struct_layout_matches_header(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "twell.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu\\n", sizeof(twell_t),'
        ' offsetof(twell_t, val), offsetof(twell_t, spill_cap), offsetof(twell_t, spill_n),'
        ' offsetof(twell_t, spill_val)); return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)],
                   check=True)
    got = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True,
                                       check=True).stdout.split()))
    S = tw.TwellStruct
    assert got == [ctypes.sizeof(S), S.val.offset, S.spill_cap.offset, S.spill_n.offset,
                   S.spill_val.offset]


def test_status_strings(lib):
    for code in range(4):
        assert tw.twell_status_string(code).startswith("TWELL_")
    assert lib.twell_version() >= 1


FAKE = 0x10000  # aligned, never dereferenced: validation fails before any device work


def _struct(T=4, F=256, tile=128, width=8, spill_cap=16, ptr=FAKE):
    return tw.TwellStruct(T, F, tile, width, ptr, ptr, ptr, ptr, spill_cap, ptr, ptr, ptr, None)


def _pack(lib, s, T=4, D=64, F=256, x=FAKE, w=FAKE, z=None):
    return lib.twell_gate_pack(x, w, T, D, F, ctypes.byref(s), z, FAKE, None)


def test_gate_pack_rejects_bad_arguments(lib):
    assert _pack(lib, _struct(), D=60) == INVALID            # D % 8
    assert _pack(lib, _struct(F=200), F=200) == INVALID      # F % 128
    assert _pack(lib, _struct(tile=64)) == INVALID           # tile
    assert _pack(lib, _struct(width=0)) == INVALID           # W
    assert _pack(lib, _struct(width=129)) == INVALID
    assert _pack(lib, _struct(T=5)) == INVALID               # T mismatch
    assert _pack(lib, _struct(), x=None) == INVALID          # null input
    assert _pack(lib, _struct(), x=FAKE + 2) == INVALID      # misaligned input
    assert _pack(lib, _struct(), z=FAKE + 4) == INVALID      # misaligned z_debug
    assert _pack(lib, _struct(spill_cap=-1)) == INVALID
    s = _struct()
    s.spill_n = None
    assert _pack(lib, s) == INVALID
    assert lib.twell_gate_pack(FAKE, FAKE, 4, 64, 256, None, None, FAKE, None) == INVALID


def test_gate_pack_empty_is_noop(lib):
    assert _pack(lib, _struct(T=0, ptr=None), T=0, x=None, w=None) == 0


def test_ffn_fwd_rejects_bad_arguments(lib):
    s = _struct()
    assert lib.twell_ffn_fwd(FAKE, ctypes.byref(s), FAKE, FAKE, 60, FAKE, FAKE, None) == INVALID
    assert lib.twell_ffn_fwd(None, ctypes.byref(s), FAKE, FAKE, 64, FAKE, FAKE, None) == INVALID
    assert lib.twell_ffn_fwd(FAKE, ctypes.byref(s), FAKE, FAKE, 64, FAKE + 8, FAKE,
                             None) == INVALID
    assert lib.twell_ffn_fwd(FAKE, None, FAKE, FAKE, 64, FAKE, FAKE, None) == INVALID
    assert lib.twell_ffn_fwd(FAKE, ctypes.byref(s), FAKE, FAKE, 256 * 13, FAKE, FAKE,
                             None) == UNSUPPORTED
    e = _struct(T=0, ptr=None)
    assert lib.twell_ffn_fwd(None, ctypes.byref(e), None, None, 64, None, None, None) == 0


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    assert _pack(lib, _struct()) in (CUDA, UNSUPPORTED)


def test_workspace_sizes(lib):
    # every workspace covers the buffers its entry point carves out of it
    # (each rounded up to 256 bytes), and bad arguments give 0
    T, D, F, C, MD = 1000, 256, 1024, 32, 64
    n_t = F // tw.TILE
    ell = T * n_t * C * 2            # one fp16 / bf16 value per ELL slot
    fd = F * D * 2                   # one 16-bit copy of a weight matrix
    fwd_tc = tw.twell_workspace_size(tw.WS_HYBRID_FWD_TC, T, D, F, C, MD)
    bwd_tc = tw.twell_workspace_size(tw.WS_HYBRID_BWD_TC, T, D, F, C, MD)
    fwd_cc = tw.twell_workspace_size(tw.WS_HYBRID_FWD, T, D, F, C, MD)
    # x rows + a + fp16 W_d, plus the dense-row buffers of the CUDA-core forward
    assert fwd_tc >= T * D * 2 + ell + fd + fwd_cc - 3 * 256
    # x rows, dy hi | lo rows, a, dz hi and lo, du, three fp16 weight copies
    assert bwd_tc >= T * D * 2 + T * 2 * D * 2 + 4 * ell + 3 * fd
    assert tw.twell_workspace_size(tw.WS_FFN_FWD_TC, 8192, 1536, 6144, 0, 0) >= \
        2 * (8192 + 1536) * 6144
    for op in (tw.WS_HYBRID_FWD, tw.WS_HYBRID_BWD, tw.WS_HYBRID_FWD_TC, tw.WS_HYBRID_BWD_TC):
        assert tw.twell_workspace_size(op, T, D, F, C, MD) > 0
        assert tw.twell_workspace_size(op, -1, D, F, C, MD) == 0
        assert tw.twell_workspace_size(op, T, 0, F, C, MD) == 0
        assert tw.twell_workspace_size(op, T, D, F, 0, MD) == 0
        assert tw.twell_workspace_size(op, T, D, F, C, -1) == 0
    assert tw.twell_workspace_size(0, T, D, F, C, MD) == 0
    # the sorted tensor-core forward adds the row order and x in that order
    assert tw.twell_workspace_size(tw.WS_FFN_FWD_TC_SORTED, 8192, 1536, 6144, 0, 0) >= \
        tw.twell_workspace_size(tw.WS_FFN_FWD_TC, 8192, 1536, 6144, 0, 0) + 8192 * (2 * 1536 + 5)
    assert tw.twell_workspace_size(7, T, D, F, C, MD) == 0
    # T = 0 needs no per-row buffers but stays a valid request
    assert tw.twell_workspace_size(tw.WS_HYBRID_BWD_TC, 0, D, F, C, MD) >= 3 * fd
