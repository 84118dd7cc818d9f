"""The C-ABI library builds, loads and exports every declared entry point; host-side
validation returns the documented error codes.  CPU only: no call here reaches a kernel."""
import ctypes
import os
import re

import pytest

import combine_topk_ids_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        moe.build()
    return moe.lib()


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for f in ("moe_workspace_size", "moe_expert_out_size", "moe_dispatch", "moe_prepare_weights",
              "moe_expert_ffn", "moe_combine", "moe_get_status", "moe_strerror"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    for f in _declared_functions():
        assert hasattr(lib, f), f


def _geom(**kw):
    base = dict(W=2, Tr=32, T=64, H=256, E=8, k=2, I=512, layout="EM", algo="LL")
    base.update(kw)
    return moe.make_geom(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(E=7), -2),                 # num_experts % world
    (dict(H=200), -3),               # hidden % 128
    (dict(I=100), -4),               # intermediate % 128
    (dict(T=65), -5),                # num_tokens > world * max_tok
    (dict(k=0), -6), (dict(k=33), -6),
    (dict(W=0), -1), (dict(layout=3), -1), (dict(algo=2), -1), (dict(quant=2), -1), (dict(expert_out=2), -1),
    (dict(W=128, E=128, Tr=1, T=1), -13),
])
def test_geometry_errors(lib, kw, code):
    g = _geom(**kw)
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(g), ctypes.byref(n)) == code
    assert moe.strerror(code) != "unknown error"


def test_workspace_size_grows_with_capacity(lib):
    a = moe.moe_workspace_size(_geom())
    b = moe.moe_workspace_size(_geom(Tr=64))
    assert 0 < a < b and a % 256 == 0
    # EXPERT_MAJOR receive buffer alone: E * W*Tr * H bf16
    assert a >= 8 * 64 * 256 * 2
    assert moe.moe_expert_out_size(_geom()) == 8 * 64 * 256 * 4
    assert moe.moe_expert_out_size(_geom(layout="RM")) == 2 * 64 * 256 * 4
    # bf16 expert_out: half the bytes, and a smaller workspace (RM/FLAT per-pick rows)
    assert moe.moe_expert_out_size(_geom(expert_out="bf16")) * 2 == moe.moe_expert_out_size(_geom())
    assert moe.moe_workspace_size(_geom(layout="RM", expert_out="bf16")) < moe.moe_workspace_size(_geom(layout="RM"))
    # FP8 rows take one byte per element (plus a float scale per 128 columns)
    f = moe.moe_workspace_size(_geom(quant="fp8"))
    assert f < a and f >= 8 * 64 * 256 + 8 * 64 * 2 * 4


def test_dispatch_host_errors_before_any_launch(lib):
    g = _geom()
    h = moe.MoeHandle()
    ws = ctypes.c_void_p(1 << 20)   # never dereferenced: every case fails validation first
    x = ctypes.c_void_p(1 << 21)
    call = lambda **kw: lib.moe_dispatch(  # noqa: E731
        ctypes.byref(kw.get("g", g)), kw.get("x", x), kw.get("ids", x), kw.get("dt", 1), None,
        kw.get("act", None), kw.get("ws", ws), kw.get("wsb", 1 << 40), ctypes.byref(h), None)
    assert call(dt=5) == -7
    assert call(ws=ctypes.c_void_p((1 << 20) + 16)) == -9
    assert call(x=ctypes.c_void_p((1 << 21) + 2)) == -9
    assert call(wsb=16) == -8
    assert call(act=ctypes.c_void_p((1 << 21) + 2)) == -9
    assert call(g=_geom(layout="RM")) == -1      # RM/FLAT need topk_weights
    assert h.magic == 0


def test_fp8_weight_calls_validate_before_launch(lib):
    g = _geom(quant="fp8")
    p = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert lib.moe_quantize_weights_fp8(ctypes.byref(g), p, p, odd, p, p, p, None) == -9
    assert lib.moe_quantize_weights_fp8(ctypes.byref(g), p, None, p, p, p, p, None) == -1
    assert lib.moe_prepare_weights_fp8(ctypes.byref(g), p, p, p, p, None) == -1   # in place
    assert lib.moe_prepare_weights_fp8(ctypes.byref(_geom(E=7, quant="fp8")), p, p, odd, odd, None) == -2


def test_calls_reject_an_unfilled_handle(lib):
    h = moe.MoeHandle()
    p = ctypes.c_void_p(1 << 20)
    assert lib.moe_expert_ffn(ctypes.byref(h), p, p, p, None) == -10
    assert lib.moe_expert_ffn_fp8(ctypes.byref(h), p, p, p, p, p, None) == -10
    assert lib.moe_selftest_wait_expiry(None, None) == -1
    assert lib.moe_combine(ctypes.byref(h), p, p, p, None) == -10
    v = ctypes.c_int32()
    assert lib.moe_get_status(ctypes.byref(h), ctypes.byref(v), None) == -10


@pytest.mark.parametrize("W,Tr,T,E,k,layout,want", [
    (2, 32, 64, 8, 2, "EM", 5),          # 128 picks, 8 experts: one routing CTA
    (8, 128, 1024, 8, 2, "EM", 5),       # 2048 picks
    (4, 1024, 4096, 16, 4, "EM", 7),     # 16384 picks: three routing kernels
    (8, 128, 1024, 256, 8, "RM", 8),     # 256 experts: three routing kernels, plus the reduction
    (4, 96, 350, 16, 4, "FLAT", 6),      # 1400 picks: one routing CTA, plus the reduction
])
def test_launches_per_layer(lib, W, Tr, T, E, k, layout, want):
    # routing (1 or 3), row scatter, GEMM1, GEMM2, RANK_MAJOR / FLAT reduction, combine
    g = moe.make_geom(W, Tr, T, 512, E, k, 256, layout, "LL")
    assert moe.moe_launches_per_layer(g) == want


def test_ctypes_structs_match_the_header(tmp_path):
    """The binding's ctypes mirrors of moe_geom and moe_handle have the C layout: a small C
    program built against include/moe.h prints sizeof and offsetof of every field."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = {"moe_geom": [n for n, _ in moe.MoeGeom._fields_],
              "moe_handle": [n for n, _ in moe.MoeHandle._fields_]}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe.h"', "int main(void) {"]
    for st, names in fields.items():
        lines.append('printf("%s sizeof %%zu\\n", sizeof(%s));' % (st, st))
        for n in names:
            lines.append('printf("%s %s %%zu\\n", offsetof(%s, %s));' % (st, n, st, n))
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        st, n, v = line.split()
        got[(st, n)] = int(v)
    for st, cls in (("moe_geom", moe.MoeGeom), ("moe_handle", moe.MoeHandle)):
        assert got[(st, "sizeof")] == ctypes.sizeof(cls), st
        for n in fields[st]:
            assert got[(st, n)] == getattr(cls, n).offset, (st, n)


def test_noalloc_validates_before_touching_a_device(lib):
    """moe_route_noalloc's host checks come first; on a host without a GB300 a valid call
    reports the device (MOE_ERR_CUDA without one, MOE_ERR_NOT_BUILT_FOR_DEVICE on another
    GPU) and never succeeds."""
    p = ctypes.c_void_p(1 << 20)
    call = lambda g, dt=1: lib.moe_route_noalloc(ctypes.byref(g), p, dt, p, p, p, p, p, p, p, None)  # noqa: E731
    assert call(_geom(layout="RM")) == -1
    assert call(_geom(), dt=5) == -7
    assert call(_geom(E=7)) == -2
    assert call(moe.make_geom(8, 16384, 8, 128, 2048, 1, 128, "EM", "LL")) == -13
    import torch
    if not torch.cuda.is_available():
        assert call(_geom()) in (-11, -12)
