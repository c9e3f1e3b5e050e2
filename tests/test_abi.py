"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/nvfp4moe.h declares, and rejects bad arguments on the host before
any launch (CPU only: no compute call reaches the device)."""
import ctypes
import os
import re

import pytest

import nvfp4_quantized_moe_token_gb300 as nv
from nvfp4_quantized_moe_token_gb300 import build as nvbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4moe.h")


@pytest.fixture(scope="module")
def L():
    nvbuild.build()
    return nv.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"NVFP4_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


def test_header_declares_the_binding_symbols():
    assert sorted(declared_functions()) == sorted(nv.SYMBOLS)


def _struct_fields(src, name):
    """Field names, in order, of `typedef struct name { ... } name;` in the header."""
    body = re.search(r"typedef struct " + name + r" \{(.*?)\} " + name + ";", src, re.S).group(1)
    return re.findall(r"(\w+)\s*;", re.sub(r"/\*.*?\*/", "", body, flags=re.S))


def test_binding_structs_and_error_bits_match_the_header():
    """The ctypes structures mirror the header field by field (a mismatch would
    shift every later field silently), and the error-word bits agree."""
    src = open(HEADER).read()
    assert _struct_fields(src, "moe_debug") == [f[0] for f in nv._Debug._fields_]
    assert _struct_fields(src, "moe_workspace_layout") == nv.LAYOUT_FIELDS
    assert _struct_fields(src, "moe_options") == [f[0] for f in nv._Options._fields_]
    assert _struct_fields(src, "nvfp4_tensor") == [f[0] for f in nv._Tensor._fields_]
    bits = dict(re.findall(r"#define NVFP4_DEVERR_(\w+) (\d+)u", src))
    assert int(bits["TIMEOUT"]) == nv.DEVERR_TIMEOUT and int(bits["BADEXPERT"]) == nv.DEVERR_BADEXPERT
    assert int(bits["BADGROUP"]) == nv.DEVERR_BADGROUP
    assert int(re.search(r"#define NVFP4_DQ_PADDED_ROWS (\d+)", src).group(1)) == nv.DQ_PADDED_ROWS


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {nv.library_path()}").read().split()
    exported = {w for w in out if not w.startswith("_") and w.islower()}
    assert set(declared_functions()) <= exported


def test_sizing_functions(L):
    assert nv.sf_bytes(16384, 2048) == 16384 * 128
    assert nv.sf_bytes(1, 16) == 128 * 4
    assert nv.sf_bytes(130, 768) == 256 * 48
    assert L.nvfp4_quantize_workspace(10, 64, 0) == 0
    assert L.nvfp4_quantize_workspace(10, 64, 1) == 256
    lay = nv.moe_workspace_layout(32768, 2048, 768, 128, 8)
    R = 32768 * 8
    assert lay["y2"] + 2 * R * 2048 <= lay["total"]
    offs = sorted(v for k, v in lay.items() if k != "total")
    assert all(o % 256 == 0 for o in offs) and len(set(offs)) == len(offs)
    assert L.moe_expert_workspace(32768, 2048, 768, 128, 8) == lay["total"]


def _t(rows, cols, ptr=4096):
    return nv._Tensor(ptr, ptr, ptr, rows, cols)


@pytest.mark.parametrize("args,code", [
    (dict(x=None), -1),
    (dict(cols=24), -2),
    (dict(mode=7), -1),
    (dict(ld=8), -1),
    (dict(x=4100), -3),
    (dict(mode=1, ws=None), -4),
])
def test_quantize_rejects_bad_arguments(L, args, code):
    a = dict(x=4096, rows=4, cols=32, ld=32, mode=0, ws=None)
    a.update(args)
    out = _t(a["rows"], a["cols"])
    rc = L.nvfp4_quantize_rows(a["x"], a["rows"], a["cols"], a["ld"], a["mode"], None, ctypes.byref(out),
                               a["ws"], 0, None)
    assert rc == code
    assert L.nvfp4_last_error().decode()


def test_linear_rejects_bad_shapes(L):
    x, w = _t(64, 96), _t(512, 96)
    assert L.nvfp4_linear(ctypes.byref(x), ctypes.byref(w), 4096, 512, None, 0, None) == -2
    x, w = _t(64, 256), _t(500, 256)
    assert L.nvfp4_linear(ctypes.byref(x), ctypes.byref(w), 4096, 512, None, 0, None) == -2
    x, w = _t(64, 256), _t(512, 128)
    assert L.nvfp4_linear(ctypes.byref(x), ctypes.byref(w), 4096, 512, None, 0, None) == -1
    x, w = _t(64, 256), _t(512, 256)
    assert L.nvfp4_linear(ctypes.byref(x), ctypes.byref(w), 4096, 500, None, 0, None) == -3


def test_moe_rejects_bad_arguments(L):
    T, H, F, E, k = 64, 2048, 768, 128, 8
    w1, w2 = _t(E * 2 * F, H), _t(E * H, F)
    opt = nv._Options(0)
    need = L.moe_expert_workspace(T, H, F, E, k)

    def call(**kw):
        a = dict(x=4096, T=T, H=H, logits=4096, E=E, k=k, w1=w1, w2=w2, F=F, out=4096, ws=4096, wsb=need)
        a.update(kw)
        return L.moe_expert_forward(a["x"], a["T"], a["H"], a["logits"], None, a["E"], a["k"],
                                    ctypes.byref(a["w1"]), ctypes.byref(a["w2"]), a["F"], ctypes.byref(opt),
                                    a["out"], None, a["ws"], a["wsb"], None)
    assert call(wsb=need - 1) == -4
    assert call(H=2000) == -2
    assert call(E=100) == -2
    assert call(k=17) == -2
    assert call(w2=_t(E * H, 2 * F)) == -1
    assert call(ws=4096 + 16) == -3
    assert call(x=None) == -1
    assert call(T=0) == -1
    for bad in (-1, 3):  # moe_options.fc2_requant outside MOE_REQUANT_AUTO .. MOE_REQUANT_IN_FC2
        opt.fc2_requant = bad
        assert call() == -1
    opt.fc2_requant = 0
    for bad in (-1, 2):  # moe_options.fc2_combine is 0 or 1
        opt.fc2_combine = bad
        assert call() == -1
    opt.fc2_combine = 0
    # the no-alloc error word's accessor refuses a null out before touching a device
    L.moe_noalloc_error_word.argtypes = [ctypes.c_void_p]
    assert L.moe_noalloc_error_word(None) == -1


def test_quantize_grouped_rejects_bad_arguments(L):
    """Host-side checks of nvfp4_quantize_grouped (no device work happens)."""
    def call(groups=4, rpg=256, cols=64, mode=1, ws=4096, wsb=64, rows=None):
        out = _t(groups * rpg if rows is None else rows, cols)
        return L.nvfp4_quantize_grouped(4096, groups, rpg, cols, mode, ctypes.byref(out), ws, wsb, None)
    assert call(mode=0) == -1            # per-tensor scales only
    assert call(groups=0) == -2
    assert call(rpg=200) == -2           # rows per group: multiples of 128
    assert call(cols=40) == -2
    assert call(rows=100) == -1          # out shape
    assert call(wsb=16 + 4 * 4 - 1) == -4
    assert call(ws=None) == -4
    assert L.nvfp4_last_error().decode()


def test_backward_gemms_reject_bad_arguments(L):
    """Host-side checks of the grouped BF16 backward GEMMs (no device work happens)."""
    for fn, nf_mult in ((L.nvfp4_grouped_dgrad_bf16, 64), (L.nvfp4_grouped_wgrad_bf16, 256)):
        def call(a=4096, b=4096, c=4096, rows=256, nf=512, kf=512, poff=None, groups=1, ws=None, wsb=0):
            return fn(a, b, c, rows, nf, kf, poff, groups, ws, wsb, None)
        assert call(a=None) == -1
        assert call(c=None) == -1
        assert call(rows=-1) == -2
        assert call(kf=320) == -2                 # output columns: multiples of 256
        assert call(nf=nf_mult + 32) == -2        # dgrad contraction / wgrad output rows
        assert call(poff=4096, groups=0) == -2
        assert call(poff=4096, groups=257) == -2
        assert call(a=4096 + 8) == -3
        assert call(ws=4098, wsb=64) == -3
        assert L.nvfp4_last_error().decode()


def test_dequantize_padded_rows_needs_offsets(L):
    t = _t(64, 256)
    assert L.nvfp4_dequantize_rows(ctypes.byref(t), nv.PER_ROW | nv.DQ_PADDED_ROWS, None, None, 0, 4096, 256,
                                   None) == -1
    assert L.nvfp4_dequantize_rows(ctypes.byref(t), 64, None, None, 0, 4096, 256, None) == -1
