"""The C ABI library on a machine without a GPU: it builds, loads, exports
every entry point include/moe.h declares, sizes workspaces, and rejects bad
arguments on the host before any CUDA call (no compute is launched here)."""

import ctypes
import math
import os
import re

import pytest

import mixture_experts_ffn_topk_gb300 as moe
from mixture_experts_ffn_topk_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")

OK, NULL, SHAPE, DTYPE, VALUE, ALIGN, WORKSPACE = 0, 1, 2, 3, 4, 5, 6
F32, BF16, F16 = 0, 1, 2
FAKE = 0x7f0000000000          # 16-byte aligned, never dereferenced
FAKE_ODD = FAKE + 8


@pytest.fixture(scope="module")
def lib():
    build.build()
    return moe.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ["moe_route", "moe_dispatch", "moe_experts_forward", "moe_combine",
              "moe_combine_add_rmsnorm", "moe_forward", "moe_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(moe.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in moe.h but not exported"
    assert sorted(moe.EXPORTED) == declared_functions()


def test_status_strings(lib):
    for code in range(11):
        assert moe.moe_status_string(code)
    assert moe.moe_status_string(99) == "unknown status"
    assert moe.moe_abi_version() == 101


def P(v):
    return ctypes.c_void_p(v)


def test_route_validation(lib):
    s = P(None)
    assert lib.moe_route(P(FAKE), 7, 4, 8, 2, 1, P(FAKE), P(FAKE), s) == DTYPE
    assert lib.moe_route(P(FAKE), F32, 4, 0, 1, 1, P(FAKE), P(FAKE), s) == SHAPE
    assert lib.moe_route(P(FAKE), F32, 4, 1025, 1, 1, P(FAKE), P(FAKE), s) == SHAPE
    assert lib.moe_route(P(FAKE), F32, 4, 8, 0, 1, P(FAKE), P(FAKE), s) == SHAPE
    assert lib.moe_route(P(FAKE), F32, 4, 8, 9, 1, P(FAKE), P(FAKE), s) == SHAPE
    assert lib.moe_route(P(FAKE), F32, -1, 8, 2, 1, P(FAKE), P(FAKE), s) == SHAPE
    assert lib.moe_route(P(None), F32, 4, 8, 2, 1, P(FAKE), P(FAKE), s) == NULL
    assert lib.moe_route(P(FAKE_ODD), F32, 4, 8, 2, 1, P(FAKE), P(FAKE), s) == ALIGN
    # T == 0 is a valid no-op even with NULL tensors
    assert lib.moe_route(P(None), BF16, 0, 8, 2, 1, P(None), P(None), s) == OK
    lib.moe_route(P(FAKE), F32, 4, 8, 9, 1, P(FAKE), P(FAKE), s)
    assert b"top_k" in lib.moe_last_error_detail()


def test_route_sigmoid_grouped_validation(lib):
    """ruDNN section 10 limits, checked on the host before any launch."""
    s = P(None)

    def call(**kw):
        a = dict(lg=P(FAKE), ldt=BF16, T=4, E=16, bias=P(FAKE), k=2, G=4, S=2, two=1, ren=1,
                 scale=2.5, idx=P(FAKE), w=P(FAKE))
        a.update(kw)
        return lib.moe_route_sigmoid_grouped(a["lg"], a["ldt"], a["T"], a["E"], a["bias"],
                                             a["k"], a["G"], a["S"], a["two"], a["ren"],
                                             a["scale"], a["idx"], a["w"], s)
    assert call(ldt=7) == DTYPE
    assert call(E=0) == SHAPE
    assert call(E=1025) == SHAPE
    assert call(G=0) == SHAPE
    assert call(G=3) == SHAPE                  # 16 % 3 != 0
    assert call(E=256, G=256) == SHAPE         # more than 128 groups
    assert call(S=0) == SHAPE
    assert call(S=5) == SHAPE                  # more than groups
    assert call(k=9) == SHAPE                  # more than S * E / G = 8
    assert call(E=128, G=1, S=1, k=65) == SHAPE    # top_k <= 64
    assert call(E=8, G=8, S=4, k=2, two=1) == SHAPE   # one expert per group
    assert call(scale=0.0) == VALUE
    assert call(scale=-1.0) == VALUE
    assert call(scale=math.inf) == VALUE
    assert call(scale=math.nan) == VALUE
    assert call(bias=P(FAKE_ODD)) == ALIGN
    assert call(lg=P(None)) == NULL
    assert call(T=0, lg=P(None), idx=P(None), w=P(None)) == OK
    call(k=9)
    assert b"top_k" in lib.moe_last_error_detail()


def test_forward_sigmoid_grouped_validation(lib):
    s = P(None)

    def call(**kw):
        a = dict(x=P(FAKE), lg=P(FAKE), bias=P(None), T=32, H=64, I=32, E=16, k=2, G=4, S=2,
                 two=0, scale=1.0, y=P(FAKE), wsb=1 << 30)
        a.update(kw)
        return lib.moe_forward_sigmoid_grouped(
            a["x"], BF16, a["lg"], BF16, a["bias"], P(FAKE), P(FAKE), P(FAKE), a["T"], a["H"],
            a["I"], a["E"], a["k"], a["G"], a["S"], a["two"], 1, a["scale"], a["y"], P(FAKE),
            a["wsb"], s)
    assert call(G=5) == SHAPE
    assert call(k=9) == SHAPE
    assert call(scale=0.0) == VALUE
    assert call(y=P(FAKE_ODD)) == ALIGN
    assert call(wsb=100) == WORKSPACE
    assert call(T=0, x=P(None), lg=P(None), y=P(None)) == OK


def _c_layout(tmp_path, ctype, fields):
    """sizeof and field offsets of a header struct as the C compiler lays it out."""
    import subprocess
    src = tmp_path / f"layout_{ctype}.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "moe.h"\n'
                   "int main(void) {\n"
                   f'    printf("%zu\\n", sizeof({ctype}));\n'
                   + "".join(f'    printf("%zu\\n", offsetof({ctype}, {n}));\n'
                             for n in fields) + "    return 0;\n}\n")
    exe = tmp_path / f"layout_{ctype}"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True)
    return [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True,
                                           text=True).stdout.split()]


@pytest.mark.parametrize("ctype,mirror", [("moe_combine_extras", "CombineExtras"),
                                          ("moe_forward_options", "ForwardOptions"),
                                          ("moe_sigmoid_grouped_routing", "SigmoidGroupedRouting"),
                                          ("moe_forward_layout", "ForwardLayout")])
def test_struct_layouts_match_header(tmp_path, ctype, mirror):
    """The binding's ctypes mirrors have the C header's layout (field offsets
    and size as the C compiler lays them out)."""
    cls = getattr(moe, mirror)
    fields = [f[0] for f in cls._fields_]
    got = _c_layout(tmp_path, ctype, fields)
    assert got[0] == ctypes.sizeof(cls)
    assert got[1:] == [getattr(cls, n).offset for n in fields]


def test_combine_v2_validation(lib):
    s = P(None)

    def call(ex=None, **kw):
        a = dict(out=P(FAKE), odt=F32, w=P(FAKE), wdt=F32, rows=P(FAKE), res=P(None),
                 gamma=P(None), gdt=F32, eps=1e-6, T=8, k=2, H=64, y=P(FAKE), dt=BF16,
                 xo=P(None), rstd=P(None))
        a.update(kw)
        return lib.moe_combine_v2(a["out"], a["odt"], a["w"], a["wdt"], a["rows"],
                                  None if ex is None else ctypes.byref(ex), a["res"], a["gamma"],
                                  a["gdt"], a["eps"], a["T"], a["k"], a["H"], a["y"], a["dt"],
                                  a["xo"], a["rstd"], s)

    def extras(**kw):
        a = dict(ids=None, E=4, zero=0, copy=0, const=0, ori=None, a1=None, a2=None, v=None,
                 shared=None, mask=None, mdims=0)
        a.update(kw)
        return moe.CombineExtras(a["ids"], a["E"], a["zero"], a["copy"], a["const"], a["ori"],
                                 a["a1"], a["a2"], a["v"], a["shared"], a["mask"], a["mdims"])
    assert call(H=60) == SHAPE
    assert call(extras(E=0)) == SHAPE
    assert call(extras(zero=-1)) == SHAPE
    assert call(extras(mdims=3)) == SHAPE
    assert call(extras(zero=1)) == NULL                     # special experts need ids
    assert call(extras(ids=FAKE, copy=1)) == NULL           # copy needs ori_x
    assert call(extras(ids=FAKE, const=1, ori=FAKE)) == NULL  # const needs alpha1/2 and V
    assert call(extras(mdims=2)) == NULL                    # mask dims without a mask
    assert call(extras(shared=FAKE_ODD)) == ALIGN
    assert call(extras(ids=FAKE, copy=1, ori=FAKE_ODD)) == ALIGN
    assert call(extras(), res=P(FAKE), gamma=P(FAKE), eps=0.0) == VALUE
    assert call(extras(), res=P(FAKE), gamma=P(FAKE)) == NULL    # norm needs x_out, rstd
    assert call(extras(), T=0, out=P(None), w=P(None), rows=P(None), y=P(None)) == OK
    assert call(None, T=0, out=P(None), w=P(None), rows=P(None), y=P(None)) == OK


def test_dispatch_special_validation(lib):
    s = P(None)
    assert lib.moe_dispatch_special(P(FAKE), 4, 2, 8, -1, P(FAKE), BF16, 64, P(FAKE), P(FAKE),
                                    P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1 << 20, s) == SHAPE
    assert lib.moe_dispatch_special(P(FAKE), 4, 2, 8, 1 << 31, P(FAKE), BF16, 64, P(FAKE),
                                    P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1 << 20,
                                    s) == SHAPE
    assert lib.moe_dispatch_special(P(None), 0, 2, 8, 3, P(None), BF16, 64, P(None), P(None),
                                    P(None), P(None), P(None), P(None), 0, s) == OK


def test_rmsnorm_validation(lib):
    s = P(None)

    def call(**kw):
        a = dict(x=P(FAKE), dt=BF16, g=P(FAKE), gdt=F32, eps=1e-6, rows=4, H=64, y=P(FAKE),
                 r=P(None))
        a.update(kw)
        return lib.moe_rmsnorm(a["x"], a["dt"], a["g"], a["gdt"], a["eps"], a["rows"], a["H"],
                               a["y"], a["r"], s)
    assert call(dt=9) == DTYPE
    assert call(gdt=F16) == DTYPE                 # gamma F32 or the input dtype
    assert call(H=60) == SHAPE
    assert call(H=16392) == SHAPE
    assert call(eps=0.0) == VALUE
    assert call(eps=math.nan) == VALUE
    assert call(x=P(None)) == NULL
    assert call(y=P(FAKE_ODD)) == ALIGN
    assert call(rows=0, x=P(None), y=P(None)) == OK


def test_dispatch_validation(lib):
    s = P(None)
    args = lambda **kw: [kw.get("idx", P(FAKE)), kw.get("T", 16), kw.get("k", 2),
                         kw.get("E", 8), kw.get("x", P(FAKE)), kw.get("xdt", BF16),
                         kw.get("H", 64), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                         kw.get("ws", P(FAKE)), kw.get("wsb", 1 << 20), s]
    assert lib.moe_dispatch(*args(xdt=5)) == DTYPE
    assert lib.moe_dispatch(*args(E=0)) == SHAPE
    assert lib.moe_dispatch(*args(H=0)) == SHAPE
    assert lib.moe_dispatch(*args(idx=P(None))) == NULL
    assert lib.moe_dispatch(*args(x=P(FAKE_ODD))) == ALIGN
    assert lib.moe_dispatch(*args(wsb=0)) == WORKSPACE
    assert lib.moe_dispatch(*args(ws=P(FAKE + 16))) == WORKSPACE
    assert lib.moe_dispatch(*args(T=0, idx=P(None))) == OK


def test_workspace_sizes(lib):
    assert lib.moe_dispatch_workspace_size(0, 2, 8) == 0
    ws = lib.moe_dispatch_workspace_size(4096, 6, 64)
    assert ws > 0 and ws % 256 == 0
    assert lib.moe_experts_workspace_size(100, 8, 64, 40, BF16) >= 100 * 40 * 2
    assert lib.moe_experts_workspace_size(100, 8, 64, 40, F32) >= 100 * 40 * 4
    # fine prefill: x_disp and h in BF16, the FP32 [T, H] combine accumulator
    fw = lib.moe_forward_workspace_size(4096, 2048, 1408, 64, 6, BF16, BF16)
    A = 4096 * 6
    assert fw >= A * (2048 * 2 + 1408 * 2) + 4096 * 2048 * 4 + A * (4 + 2 + 4 + 4)
    # coarse prefill (accumulator past 64 MiB): FP32 expert outputs [T*k, H]
    fw = lib.moe_forward_workspace_size(16384, 4096, 14336, 8, 2, BF16, F32)
    A = 16384 * 2
    assert fw >= A * (4096 * 2 + 14336 * 2 + 4096 * 4)
    assert lib.moe_forward_workspace_size(4096, 2048, 1408, 64, 65, BF16, BF16) == 0


def test_experts_validation(lib):
    s = P(None)
    base = dict(x=P(FAKE), off=P(FAKE), rows=64, g=P(FAKE), u=P(FAKE), d=P(FAKE),
                E=4, H=64, I=32, dt=BF16, out=P(FAKE), ws=P(FAKE), wsb=1 << 20)

    def call(**kw):
        a = dict(base, **kw)
        return lib.moe_experts_forward(a["x"], a["off"], a["rows"], a["g"], a["u"],
                                       a["d"], a["E"], a["H"], a["I"], a["dt"],
                                       a["out"], a.get("odt", a["dt"]), a["ws"], a["wsb"], s)
    assert call(dt=9) == DTYPE
    assert call(odt=F16) == DTYPE       # output must be the expert dtype or F32
    assert call(H=60) == SHAPE          # 60 * 2 bytes is not a 16-byte multiple
    assert call(I=6, dt=F32) == SHAPE   # 24 bytes
    assert call(E=2000) == SHAPE
    assert call(g=P(None)) == NULL
    assert call(d=P(FAKE_ODD)) == ALIGN
    assert call(wsb=16) == WORKSPACE
    assert call(rows=0, x=P(None)) == OK


def test_combine_validation(lib):
    s = P(None)
    assert lib.moe_combine(P(FAKE), BF16, P(FAKE), F32, P(FAKE), 8, 2, 60, P(FAKE), BF16, s) == SHAPE
    assert lib.moe_combine(P(FAKE), 4, P(FAKE), F32, P(FAKE), 8, 2, 64, P(FAKE), BF16, s) == DTYPE
    assert lib.moe_combine(P(FAKE), F16, P(FAKE), F32, P(FAKE), 8, 2, 64, P(FAKE), BF16, s) == DTYPE
    assert lib.moe_combine(P(None), BF16, P(FAKE), F32, P(FAKE), 8, 2, 64, P(FAKE), BF16, s) == NULL
    assert lib.moe_combine(P(FAKE), F32, P(FAKE), F32, P(FAKE), 8, 2, 64, P(FAKE_ODD), BF16, s) == ALIGN
    assert lib.moe_combine(P(FAKE), BF16, P(FAKE), F32, P(FAKE), 0, 2, 64, P(None), BF16, s) == OK
    for eps in (0.0, -1e-6, math.inf, math.nan):
        rc = lib.moe_combine_add_rmsnorm(P(FAKE), BF16, P(FAKE), F32, P(FAKE), P(FAKE), BF16,
                                         P(FAKE), BF16, eps, 8, 2, 64, P(FAKE), P(FAKE),
                                         P(FAKE), s)
        assert rc == VALUE, eps
    big = 8 * 256 * 8 + 8
    assert lib.moe_combine_add_rmsnorm(P(FAKE), BF16, P(FAKE), F32, P(FAKE), P(FAKE), BF16,
                                       P(FAKE), BF16, 1e-6, 8, 2, big, P(FAKE), P(FAKE),
                                       P(FAKE), s) == SHAPE


def test_forward_validation(lib):
    s = P(None)

    def call(**kw):
        a = dict(x=P(FAKE), dt=BF16, lg=P(FAKE), ldt=BF16, T=32, H=64, I=32, E=8, k=2,
                 y=P(FAKE), ws=P(FAKE), wsb=1 << 30)
        a.update(kw)
        return lib.moe_forward(a["x"], a["dt"], a["lg"], a["ldt"], P(FAKE), P(FAKE),
                               P(FAKE), a["T"], a["H"], a["I"], a["E"], a["k"], 1,
                               a["y"], a["ws"], a["wsb"], s)
    assert call(ldt=3) == DTYPE
    assert call(k=9) == SHAPE
    assert call(k=0) == SHAPE
    assert call(lg=P(None)) == NULL
    assert call(y=P(FAKE_ODD)) == ALIGN
    assert call(wsb=100) == WORKSPACE
    assert call(T=0, x=P(None), lg=P(None), y=P(None)) == OK


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        moe.moe_route(torch.zeros(4, 8), 2, True, stream=0)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        moe.load_library(str(tmp_path / "nope.so"))


def test_training_validation(lib):
    """First-order training entry points (ruDNN user guide, section 12):
    every bad argument is refused on the host, before any CUDA call."""
    P = ctypes.c_void_p
    st = P(None)
    U32, I32, I64 = 0, 1, 2

    def rw(**kw):
        a = dict(lg=P(FAKE), ldt=F32, T=8, E=16, idx=P(FAKE), idt=I32, k=4, sc=0, rn=1,
                 scale=1.0, w=P(FAKE))
        a.update(kw)
        return lib.moe_router_weights(a["lg"], a["ldt"], a["T"], a["E"], a["idx"], a["idt"],
                                      a["k"], a["sc"], a["rn"], a["scale"], a["w"], st)

    assert rw(ldt=5) == DTYPE
    assert rw(idt=3) == DTYPE
    assert rw(sc=2) == DTYPE
    assert rw(E=0) == SHAPE
    assert rw(E=1025) == SHAPE
    assert rw(k=17) == SHAPE                       # k > E
    assert rw(E=100, k=65) == SHAPE                # k > 64
    for bad in (0.0, -1.0, math.inf, math.nan):
        assert rw(scale=bad) == VALUE
    assert rw(lg=P(None)) == NULL
    assert rw(w=P(FAKE_ODD)) == ALIGN
    assert rw(T=0, lg=P(None), idx=P(None), w=P(None)) == OK

    def rb(**kw):
        a = dict(lg=P(FAKE), ldt=BF16, T=8, E=16, idx=P(FAKE), idt=I64, k=4, gw=P(FAKE), sc=1,
                 rn=0, scale=2.0, dl=P(FAKE))
        a.update(kw)
        return lib.moe_router_backward(a["lg"], a["ldt"], a["T"], a["E"], a["idx"], a["idt"],
                                       a["k"], a["gw"], a["sc"], a["rn"], a["scale"], a["dl"], st)

    assert rb(idt=U32, sc=3) == DTYPE
    assert rb(gw=P(None)) == NULL
    assert rb(dl=P(FAKE_ODD)) == ALIGN
    assert rb(scale=math.inf) == VALUE
    assert rb(T=0, lg=P(None), idx=P(None), gw=P(None), dl=P(None)) == OK

    def cb(**kw):
        a = dict(out=P(FAKE), odt=F32, w=P(FAKE), wdt=F32, rows=P(FAKE), gy=P(FAKE), T=8, k=2,
                 H=64, dt=BF16, dexp=P(FAKE), dw=P(FAKE))
        a.update(kw)
        return lib.moe_combine_backward(a["out"], a["odt"], a["w"], a["wdt"], a["rows"], a["gy"],
                                        a["T"], a["k"], a["H"], a["dt"], a["dexp"], a["dw"], st)

    assert cb(odt=F16) == DTYPE                    # outputs neither the dtype nor F32
    assert cb(H=60) == SHAPE
    assert cb(k=0) == SHAPE
    assert cb(dw=P(None)) == NULL
    assert cb(gy=P(FAKE_ODD)) == ALIGN
    assert cb(T=0, out=P(None), w=P(None), rows=P(None), gy=P(None), dexp=P(None),
              dw=P(None)) == OK

    assert lib.moe_dispatch_backward(P(FAKE), 7, P(FAKE), 8, 2, 64, P(FAKE), st) == DTYPE
    assert lib.moe_dispatch_backward(P(FAKE), BF16, P(FAKE), 8, 2, 60, P(FAKE), st) == SHAPE
    assert lib.moe_dispatch_backward(P(None), BF16, P(FAKE), 8, 2, 64, P(FAKE), st) == NULL
    assert lib.moe_dispatch_backward(P(None), BF16, P(None), 0, 2, 64, P(None), st) == OK

    # training forward: the cache replaces the workspace
    need = lib.moe_experts_training_cache_size(100, 64, BF16)
    assert need == math.ceil(100 * 64 * (2 + 8) / 256) * 256
    assert lib.moe_experts_training_cache_size(100, 64, F32) == math.ceil(100 * 64 * 12 / 256) * 256

    def ft(**kw):
        a = dict(rows=100, E=4, H=64, I=64, dt=BF16, odt=F32, cache=P(FAKE), nb=need)
        a.update(kw)
        return lib.moe_experts_forward_training(P(FAKE), P(FAKE), a["rows"], P(FAKE), P(FAKE),
                                                P(FAKE), a["E"], a["H"], a["I"], a["dt"],
                                                P(FAKE), a["odt"], a["cache"], a["nb"], st)

    assert ft(odt=F16) == DTYPE
    assert ft(H=60) == SHAPE
    assert ft(nb=need - 256) == WORKSPACE
    assert ft(cache=P(FAKE + 16)) == WORKSPACE       # not 256-byte aligned
    assert ft(rows=0) == OK

    # backward: dg | du [rows, 2I] and, for 16-bit types, per-expert TMA maps
    ws = lib.moe_experts_backward_workspace_size(100, 4, 64, 64, BF16)
    assert ws >= 2 * 100 * 64 * 2 + 4 * 5 * 128
    assert lib.moe_experts_backward_workspace_size(100, 4, 64, 64, F32) == \
        math.ceil(2 * 100 * 64 * 4 / 256) * 256
    assert lib.moe_experts_backward_workspace_size(0, 4, 64, 64, BF16) > 0

    def bw(**kw):
        a = dict(rows=100, dt=BF16, ws=P(FAKE), nb=ws, gg=P(FAKE))
        a.update(kw)
        return lib.moe_experts_backward(P(FAKE), P(FAKE), a["rows"], P(FAKE), P(FAKE), P(FAKE),
                                        4, 64, 64, a["dt"], P(FAKE), P(FAKE), P(FAKE), a["gg"],
                                        P(FAKE), P(FAKE), a["ws"], a["nb"], st)

    assert bw(dt=9) == DTYPE
    assert bw(gg=P(None)) == NULL
    assert bw(nb=ws - 256) == WORKSPACE
    assert bw(rows=0, ws=P(None), nb=0) == WORKSPACE   # the maps are needed without rows too


def test_forward_ex_validation(lib):
    s = P(None)

    def call(flags=0, **kw):
        a = dict(x=P(FAKE), dt=BF16, lg=P(FAKE), ldt=BF16, T=32, H=64, I=32, E=8, k=2,
                 y=P(FAKE), ws=P(FAKE), wsb=1 << 30)
        a.update(kw)
        opt = moe.ForwardOptions()
        opt.flags = flags
        return lib.moe_forward_ex(a["x"], a["dt"], a["lg"], a["ldt"], P(FAKE), P(FAKE),
                                  P(FAKE), a["T"], a["H"], a["I"], a["E"], a["k"], 1,
                                  a["y"], a["ws"], a["wsb"], ctypes.byref(opt), s)
    assert call(flags=2) == VALUE            # unknown option bit
    assert call(ldt=3) == DTYPE
    assert call(k=9) == SHAPE
    assert call(lg=P(None)) == NULL
    assert call(y=P(FAKE_ODD)) == ALIGN
    # the deterministic forward needs the larger workspace
    need = lib.moe_forward_workspace_size_ex(32, 64, 32, 8, 2, BF16, BF16, 1)
    assert need > lib.moe_forward_workspace_size_ex(32, 64, 32, 8, 2, BF16, BF16, 0)
    assert call(flags=1, wsb=lib.moe_forward_workspace_size(32, 64, 32, 8, 2, BF16, BF16)) \
        == WORKSPACE
    assert call(flags=1, T=0, x=P(None), lg=P(None), y=P(None)) == OK
    # sigmoid routing limits through the options
    sg = moe.SigmoidGroupedRouting(None, 3, 1, 0, 1.0)      # 3 groups do not divide E = 8
    opt = moe.ForwardOptions()
    opt.sigmoid_grouped = ctypes.pointer(sg)
    rc = lib.moe_forward_ex(P(FAKE), BF16, P(FAKE), BF16, P(FAKE), P(FAKE), P(FAKE), 32, 64, 32,
                            8, 2, 1, P(FAKE), P(FAKE), 1 << 30, ctypes.byref(opt), s)
    assert rc == SHAPE


def test_forward_workspace_layout(lib):
    """The layout names disjoint, 256-byte aligned regions of the workspace,
    in the sizes the header gives them, and its total is the workspace size."""
    for (T, H, I, E, k, dt, ldt) in [(4096, 2048, 1408, 64, 6, BF16, BF16),
                                     (16384, 4096, 14336, 8, 2, BF16, F32),
                                     (128, 7168, 2048, 256, 8, BF16, F32),
                                     (64, 128, 256, 8, 2, F32, F32)]:
        for flags in (0, 1):
            lay = moe.ForwardLayout()
            assert lib.moe_forward_workspace_layout(T, H, I, E, k, dt, ldt, flags,
                                                    ctypes.byref(lay)) == OK
            assert lay.total == lib.moe_forward_workspace_size_ex(T, H, I, E, k, dt, ldt, flags)
            A, eb, lb = T * k, (4 if dt == F32 else 2), (4 if ldt == F32 else 2)
            regions = sorted([(lay.expert_indices, A * 4), (lay.weights, A * lb),
                              (lay.counts, E * 4), (lay.offsets, (E + 1) * 4),
                              (lay.row_of, A * 4), (lay.src_of, A * 4),
                              (lay.x_disp, A * H * eb)])
            for (a, n), (b, _) in zip(regions, regions[1:]):
                assert a % 256 == 0 and a + n <= b
            assert regions[-1][0] + regions[-1][1] <= lay.total
    lay = moe.ForwardLayout()
    assert lib.moe_forward_workspace_layout(8, 64, 32, 8, 2, BF16, BF16, 4,
                                            ctypes.byref(lay)) == VALUE
    assert lib.moe_forward_workspace_layout(8, 64, 32, 8, 9, BF16, BF16, 0,
                                            ctypes.byref(lay)) == SHAPE
    assert lib.moe_forward_workspace_layout(8, 64, 32, 8, 2, BF16, BF16, 0, None) == NULL


def test_wait_limit_setting(lib):
    assert lib.moe_wait_limit_ns() == 2_000_000_000
    try:
        assert lib.moe_set_wait_limit_ns(5_000_000) == OK
        assert lib.moe_wait_limit_ns() == 5_000_000
        assert lib.moe_set_wait_limit_ns(61_000_000_000) == VALUE
        assert lib.moe_wait_limit_ns() == 5_000_000
    finally:
        assert lib.moe_set_wait_limit_ns(0) == OK
    assert lib.moe_wait_limit_ns() == 2_000_000_000


def test_selftest_wait_expiry_validation(lib):
    s = P(None)
    need = lib.moe_selftest_wait_expiry_workspace_size(2, 300, 256, 128)
    assert need >= 2 * 256 * 128 * 2 + 600 * 128 * 2
    assert lib.moe_selftest_wait_expiry_workspace_size(0, 300, 256, 128) == 0
    assert lib.moe_selftest_wait_expiry(0, 300, 256, 128, P(FAKE), P(FAKE), need, s) == SHAPE
    assert lib.moe_selftest_wait_expiry(2, 300, 250, 128, P(FAKE), P(FAKE), need, s) == SHAPE
    assert lib.moe_selftest_wait_expiry(2, 300, 256, 128, P(None), P(FAKE), need, s) == NULL
    assert lib.moe_selftest_wait_expiry(2, 300, 256, 128, P(FAKE_ODD), P(FAKE), need, s) == ALIGN
    assert lib.moe_selftest_wait_expiry(2, 300, 256, 128, P(FAKE), P(FAKE), need - 1, s) == WORKSPACE


def test_dispatch_noalloc_validation_order(lib):
    """The no-alloc dispatch checks its arguments as moe_dispatch does before
    it tests the size against its built-in scratch."""
    s = P(None)
    args = lambda **kw: [kw.get("idx", P(FAKE)), kw.get("T", 262144), kw.get("k", 8),
                         kw.get("E", 1024), kw.get("x", P(FAKE)), kw.get("xdt", BF16),
                         kw.get("H", 8), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), s]
    # oversized (1-2 MiB of chunk counts, depending on the SM count the chunk
    # size follows) and a bad dtype / pointer: the argument's own status
    # comes first
    assert lib.moe_dispatch_noalloc(*args(xdt=7)) == DTYPE
    assert lib.moe_dispatch_noalloc(*args(idx=P(None))) == NULL
    assert lib.moe_dispatch_noalloc(*args(x=P(FAKE_ODD))) == ALIGN
    assert lib.moe_dispatch_noalloc(*args(E=0)) == SHAPE
    assert lib.moe_dispatch_workspace_size(262144, 8, 1024) > 256 * 1024
    assert lib.moe_dispatch_noalloc(*args()) == WORKSPACE
    assert lib.moe_dispatch_noalloc(*args(T=0, idx=P(None))) == OK


def test_bounds_build_flag_rule():
    """MOE_DEBUG_BOUNDS: unset, empty or 0 loads the normal library, 1 the
    bounds-checking one, anything else is an error."""
    assert moe.library_path({}) == moe.LIB_PATH
    assert moe.library_path({"MOE_DEBUG_BOUNDS": "0"}) == moe.LIB_PATH
    assert moe.library_path({"MOE_DEBUG_BOUNDS": ""}) == moe.LIB_PATH
    assert moe.library_path({"MOE_DEBUG_BOUNDS": "1"}) == moe.LIB_PATH_DEBUG
    for bad in ("2", "yes", "true", " 1"):
        with pytest.raises(ValueError):
            moe.library_path({"MOE_DEBUG_BOUNDS": bad})


def test_bounds_build_exports_the_same_abi():
    path = build.build(debug_bounds=True)
    raw = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(raw, name), name
