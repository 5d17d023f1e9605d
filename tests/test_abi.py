"""The C-ABI library loads without a GPU and exports every function include/dm.h
declares; host-side argument validation answers before any CUDA call."""
import ctypes
import os
import re

import pytest

import fp8_attention_gb300 as dm
from fp8_attention_gb300 import build as dm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dm.h")


@pytest.fixture(scope="module")
def lib():
    dm_build.build()
    return dm.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(dm_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("dm_quantize", "dm_attn_fwd", "dm_attn_delta", "dm_attn_bwd", "dm_attn_bwd_workspace_size",
              "dm_get_status", "dm_status_string"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    assert dm.dm_version() == 100
    for code, name in ((0, "DM_OK"), (2, "DM_ERR_SHAPE"), (7, "DM_ERR_TIMEOUT")):
        assert dm.dm_status_string(code) == name
    assert dm.dm_status_string(99) == "DM_ERR_UNKNOWN"


def test_knobs(lib):
    assert lib.dm_set_knob(0, -1) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_set_knob(7, 1) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_set_knob(dm.DM_KNOB_WAIT_LIMIT_NS, 0) == 0


def _p(B=1, Hq=2, Hkv=1, N=256, d=64, causal=1, scale=0.0, d_v=0, kv_offset=0, kv_len=0):
    return dm._Params(B, Hq, Hkv, N, d, causal, scale, d_v, kv_offset, kv_len)


def test_validation_without_gpu(lib):
    """Every check below fails before the library touches the CUDA runtime."""
    A = 0x10000  # aligned fake device addresses: never dereferenced by these calls
    f = dm._Fp8(A, A)
    fwd = lib.dm_attn_fwd
    assert fwd(None, f, f, f, A, 0, A, None) == dm.DM_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_p(d=96)), f, f, f, A, 0, A, None) == dm.DM_ERR_SHAPE
    # value head dimension: d != d_v only with both in {128, 192, 256}
    for d, d_v in ((192, 64), (64, 128), (128, 96), (320, 128), (192, 320)):
        assert fwd(ctypes.byref(_p(d=d, d_v=d_v)), f, f, f, A, 0, A, None) == dm.DM_ERR_SHAPE, (d, d_v)
    for d, d_v in ((192, 128), (256, 128), (128, 256), (192, 0), (192, 192)):
        # passes the shape checks; stopped here by the bad dtype that follows them
        assert fwd(ctypes.byref(_p(d=d, d_v=d_v)), f, f, f, A, 5, A, None) == dm.DM_ERR_DTYPE, (d, d_v)
    assert fwd(ctypes.byref(_p(Hq=3, Hkv=2)), f, f, f, A, 0, A, None) == dm.DM_ERR_SHAPE
    assert fwd(ctypes.byref(_p(N=-1)), f, f, f, A, 0, A, None) == dm.DM_ERR_SHAPE
    assert fwd(ctypes.byref(_p(B=1 << 20, Hq=64, Hkv=1, N=1 << 10, d=128)), f, f, f, A, 0, A, None) \
        == dm.DM_ERR_SHAPE
    assert fwd(ctypes.byref(_p()), f, f, f, A, 5, A, None) == dm.DM_ERR_DTYPE
    assert fwd(ctypes.byref(_p()), dm._Fp8(A + 1, A), f, f, A, 0, A, None) == dm.DM_ERR_ALIGNMENT
    assert fwd(ctypes.byref(_p()), dm._Fp8(None, A), f, f, A, 0, A, None) == dm.DM_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_p(scale=float("nan"))), f, f, f, A, 0, A, None) == dm.DM_ERR_INVALID_ARG
    # empty problems are valid no-ops, even with NULL pointers
    z = dm._Fp8(None, None)
    assert fwd(ctypes.byref(_p(B=0)), z, z, z, None, 0, None, None) == 0
    assert fwd(ctypes.byref(_p(N=0)), z, z, z, None, 0, None, None) == 0
    assert lib.dm_quantize(None, 0, 0, 2, 128, 64, 0, None, None, None, None) == 0
    assert lib.dm_quantize(A, 2, 1, 2, 128, 64, 0, A, A, None, None) == dm.DM_ERR_DTYPE
    assert lib.dm_quantize(A, 0, 1, 2, 128, 64, 2, A, A, None, None) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_quantize(A, 0, 1, 2, 128, 32, 0, A, A, None, None) == dm.DM_ERR_SHAPE
    J = dm._QuantJob
    two = (J * 2)(J(A, 1, 2, 128, 64, 0, A, A, None), J(A, 1, 2, 128, 128, 1, A, A, None))
    assert lib.dm_quantize_batch(two, 2, 0, None) == dm.DM_ERR_SHAPE           # d differs between jobs
    assert lib.dm_quantize_batch(two, 9, 0, None) == dm.DM_ERR_INVALID_ARG     # more than 8 jobs
    assert lib.dm_quantize_batch(None, 1, 0, None) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_quantize_batch(two, 1, 5, None) == dm.DM_ERR_DTYPE
    bad = (J * 1)(J(A + 4, 1, 2, 128, 64, 0, A, A, None))
    assert lib.dm_quantize_batch(bad, 1, 0, None) == dm.DM_ERR_ALIGNMENT
    empty = (J * 1)(J(None, 0, 2, 128, 64, 0, None, None, None))
    assert lib.dm_quantize_batch(empty, 1, 0, None) == 0
    assert lib.dm_quantize_batch(None, 0, 0, None) == 0
    assert lib.dm_attn_delta(ctypes.byref(_p()), 3, f, f, f, f, A, A, 0, A, 0, A, None) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_attn_delta(ctypes.byref(_p()), 1, f, f, f, f, A, None, 0, A, 0, A, None) \
        == dm.DM_ERR_INVALID_ARG
    bwd = lib.dm_attn_bwd
    assert bwd(ctypes.byref(_p()), 0, f, f, f, f, A, None, None, 0, None, 0, A, A, A, None, A, 16, None) \
        == dm.DM_ERR_INVALID_ARG  # workspace too small for the internally computed delta


def test_noalloc_validates_like_the_workspace_backward(lib):
    """dm_attn_bwd_noalloc answers a bad call with the status dm_attn_bwd gives
    it, also when the problem is empty (B = 0 or N = 0), before any CUDA call."""
    A = 0x10000
    f = dm._Fp8(A, A)
    z = dm._Fp8(None, None)

    def both(params, mode, ff):
        na = lib.dm_attn_bwd_noalloc(ctypes.byref(params), mode, ff, ff, ff, ff, A, None, 0, None, 0, A, A, A,
                                     None, None)
        ws = lib.dm_attn_bwd(ctypes.byref(params), mode, ff, ff, ff, ff, A, None, None, 0, None, 0, A, A, A,
                             None, A, 1 << 30, None)
        return na, ws

    for params, mode, ff, want in ((_p(B=0, d=100), 0, z, dm.DM_ERR_SHAPE),
                                   (_p(N=0, Hq=3, Hkv=2), 0, z, dm.DM_ERR_SHAPE),
                                   (_p(B=0), 7, z, dm.DM_ERR_INVALID_ARG),
                                   (_p(B=0, scale=float("inf")), 0, z, dm.DM_ERR_INVALID_ARG),
                                   (_p(B=0), 0, z, dm.DM_OK),
                                   (_p(d=96), 0, f, dm.DM_ERR_SHAPE)):
        assert both(params, mode, ff) == (want, want), (params.B, params.N, params.d, mode)
    assert lib.dm_attn_bwd_noalloc(None, 0, f, f, f, f, A, None, 0, None, 0, A, A, A, None, None) \
        == dm.DM_ERR_INVALID_ARG


def test_key_block_validation_without_gpu(lib):
    """Key blocks: a 128-aligned start inside the sequence; the backward of a
    block needs the merged delta; the merges reject bad part counts and dtypes."""
    A = 0x10000
    f = dm._Fp8(A, A)
    fwd = lib.dm_attn_fwd
    for off, ln in ((64, 0), (-128, 0), (256, 0), (128, 129), (0, -1)):
        p = _p(N=256, kv_offset=off, kv_len=ln)
        assert fwd(ctypes.byref(p), f, f, f, A, 5, A, None) == dm.DM_ERR_SHAPE, (off, ln)
    for off, ln in ((128, 0), (128, 128), (0, 128), (0, 256)):
        p = _p(N=256, kv_offset=off, kv_len=ln)   # valid: stopped by the bad dtype after the shape checks
        assert fwd(ctypes.byref(p), f, f, f, A, 5, A, None) == dm.DM_ERR_DTYPE, (off, ln)
    blk = _p(N=256, kv_offset=128)
    assert lib.dm_attn_bwd(ctypes.byref(blk), 0, f, f, f, f, A, None, None, 0, None, 0, A, A, A, None, A, 1 << 20,
                           None) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_attn_bwd_noalloc(ctypes.byref(blk), 0, f, f, f, f, A, None, 0, None, 0, A, A, A, None,
                                   None) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_attn_merge(ctypes.byref(_p()), 0, A, A, A, 0, A, None) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_attn_merge(ctypes.byref(_p()), 2, A, A, A, 4, A, None) == dm.DM_ERR_DTYPE
    assert lib.dm_attn_merge(ctypes.byref(_p()), 2, A + 4, A, A, 0, A, None) == dm.DM_ERR_ALIGNMENT
    assert lib.dm_attn_merge(ctypes.byref(_p(B=0)), 2, None, None, None, 0, None, None) == 0
    assert lib.dm_attn_delta_combine(ctypes.byref(_p()), 0, A, A, A, None) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_attn_delta_combine(ctypes.byref(_p()), 1, A, None, A, None) == dm.DM_ERR_INVALID_ARG
    assert lib.dm_attn_delta_partial(ctypes.byref(_p()), f, f, f, f, A, A, None, None) == dm.DM_ERR_INVALID_ARG


def test_workspace_size(lib):
    assert dm.dm_attn_bwd_workspace_size(dm.AttnParams(2, 4, 2, 1000, 64)) == ((2 * 4 * 1000 * 4 + 255) // 256) * 256
    assert dm.dm_attn_bwd_workspace_size(dm.AttnParams(2, 4, 3, 1000, 64)) == 0


def test_prologue_validation_without_gpu(lib):
    """dm_qk_prologue_batch and dm_rope_table reject bad arguments before any CUDA call."""
    A = 0x10000
    J = dm._PrologueJob
    ok = J(A, 1, 2, 256, 128, A, A, A, A, A)
    one = (J * 1)(ok)
    pro = lib.dm_qk_prologue_batch
    assert pro(one, 1, 5, 1e-6, None) == dm.DM_ERR_DTYPE
    assert pro(one, 5, 0, 1e-6, None) == dm.DM_ERR_INVALID_ARG          # more than 4 jobs
    assert pro(one, 1, 0, 0.0, None) == dm.DM_ERR_INVALID_ARG           # eps must be > 0
    assert pro(one, 1, 0, float("inf"), None) == dm.DM_ERR_INVALID_ARG
    assert pro(None, 1, 0, 1e-6, None) == dm.DM_ERR_INVALID_ARG
    assert pro((J * 1)(J(A, 1, 2, 256, 96, A, A, A, A, A)), 1, 0, 1e-6, None) == dm.DM_ERR_SHAPE
    two = (J * 2)(ok, J(A, 1, 2, 256, 64, A, A, A, A, A))
    assert pro(two, 2, 0, 1e-6, None) == dm.DM_ERR_SHAPE                # d differs between jobs
    assert pro((J * 1)(J(A, 1, 2, 256, 128, A, A, None, A, A)), 1, 0, 1e-6, None) == dm.DM_ERR_INVALID_ARG
    assert pro((J * 1)(J(A + 8, 1, 2, 256, 128, A, A, A, A, A)), 1, 0, 1e-6, None) == dm.DM_ERR_ALIGNMENT
    assert pro((J * 1)(J(A, 1, 2, 256, 128, A + 4, A, A, A, A)), 1, 0, 1e-6, None) == dm.DM_ERR_ALIGNMENT
    assert pro((J * 1)(J(A, 1, 2, 256, 128, A, A + 4, A + 4, A, A)), 1, 0, 1e-6, None) == dm.DM_ERR_ALIGNMENT
    assert pro((J * 1)(J(None, 0, 2, 256, 128, None, None, None, None, None)), 1, 0, 1e-6, None) == 0
    assert pro(None, 0, 0, 1e-6, None) == 0
    rt = lib.dm_rope_table
    assert rt(16, 12, 1e4, A, A, None) == dm.DM_ERR_SHAPE               # d not a multiple of 8
    assert rt(-1, 64, 1e4, A, A, None) == dm.DM_ERR_SHAPE
    assert rt(16, 64, 1.0, A, A, None) == dm.DM_ERR_INVALID_ARG         # base must exceed 1
    assert rt(16, 64, 1e4, None, A, None) == dm.DM_ERR_INVALID_ARG
    assert rt(16, 64, 1e4, A + 4, A, None) == dm.DM_ERR_ALIGNMENT
    assert rt(0, 64, 1e4, None, None, None) == 0


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/dm.h compiles as strict C99 (no C++ or torch types) and a C
    program links against libdm.so and calls host-only entry points."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "abi.c"
    src.write_text(
        '#include "dm.h"\n#include <stdio.h>\n'
        "int main(void) {\n"
        "  dm_quantize_job qj = {0};\n  dm_prologue_job pj = {0};\n  (void)qj; (void)pj;\n"
        '  printf("%d %s\\n", dm_version(), dm_status_string(DM_ERR_SHAPE));\n'
        "  return dm_quantize_batch(NULL, 0, DM_BF16, NULL) == DM_OK ? 0 : 1;\n}\n")
    libdir = os.path.dirname(dm.LIB_PATH)
    exe = tmp_path / "abi"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-L", libdir, "-ldm", f"-Wl,-rpath,{libdir}", "-o", str(exe)]
    subprocess.run(cmd, check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    assert out.split() == ["100", "DM_ERR_SHAPE"]
