"""The C ABI without a GPU: the library builds, loads, exports every function
include/attn.h declares, and rejects bad arguments on the host before it
touches a device."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_attn_gb300 import build as B
    B.build()
    from exact_attention_attn_gb300.binding import load_library
    return load_library()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names.update(re.findall(r"ATTN_API\s+[\w\s\*]*?\b(attn_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"attn_fwd", "attn_fwd_splitkv", "attn_fwd_plan", "attn_fwd_status", "attn_strerror", "attn_version"} <= names
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert names <= exported
    # nothing else leaks out of the library's C ABI namespace
    assert {n for n in exported if n.startswith("attn_")} == names


def test_version_and_strerror(lib):
    assert lib.attn_version() == 100
    for code in range(0, -9, -1):
        assert lib.attn_strerror(code)
    assert b"unknown" in lib.attn_strerror(-99)


class Buf:
    """16-byte aligned host addresses; never dereferenced (argument checks
    return before any device work)."""
    def __init__(self):
        self.raw = ctypes.create_string_buffer(256)
        base = ctypes.addressof(self.raw)
        self.p = (base + 15) & ~15


def call(lib, q, k, v, o, l, B=1, Hq=2, Hkv=1, Nq=8, Nkv=8, D=64, scale=0.125, causal=0):
    return lib.attn_fwd(q, k, v, o, l, B, Hq, Hkv, Nq, Nkv, D, scale, causal, None)


def test_argument_errors(lib):
    b = Buf()
    p = b.p
    ARG, ALIGN = -1, -2
    assert call(lib, p, p, p, p, p, D=65) == ARG
    assert call(lib, p, p, p, p, p, D=32) == ARG
    assert call(lib, p, p, p, p, p, D=1088) == ARG
    assert call(lib, p, p, p, p, p, Hq=3, Hkv=2) == ARG
    assert call(lib, p, p, p, p, p, Hkv=0) == ARG
    assert call(lib, p, p, p, p, p, B=-1) == ARG
    assert call(lib, p, p, p, p, p, Nq=-5) == ARG
    assert call(lib, p, p, p, p, p, scale=float("nan")) == ARG
    assert call(lib, p, p, p, p, p, scale=float("inf")) == ARG
    assert call(lib, p, p, p, p, p, causal=2) == ARG
    assert call(lib, None, p, p, p, p) == ARG
    assert call(lib, p, None, p, p, p) == ARG
    assert call(lib, p, p, p, p, None) == ARG
    assert call(lib, p + 2, p, p, p, p) == ALIGN
    assert call(lib, p, p, p + 8, p, p) == ALIGN
    assert call(lib, p, p, p, p, p + 4) == ALIGN
    # empty problems succeed without touching a device
    assert call(lib, None, None, None, None, None, B=0) == 0
    assert call(lib, None, None, None, None, None, Nq=0) == 0


def test_splitkv_argument_errors(lib):
    import ctypes as C
    lib.attn_fwd_splitkv.argtypes = [C.c_void_p] * 5 + [C.c_int] * 6 + [C.c_float, C.c_int, C.c_int, C.c_void_p]
    b = Buf()
    p = b.p
    assert lib.attn_fwd_splitkv(p, p, p, p, p, 1, 2, 1, 8, 8, 64, 0.125, 0, -1, None) == -1
    assert lib.attn_fwd_splitkv(p, p, p, p, p, 1, 2, 1, 8, 8, 64, 0.125, 0, 65, None) == -1
    assert lib.attn_fwd_splitkv(p, p, p, p, p, 1, 2, 1, 8, 8, 65, 0.125, 0, 2, None) == -1
    assert lib.attn_fwd_splitkv(None, None, None, None, None, 0, 2, 1, 8, 8, 64, 0.125, 0, 2, None) == 0


def test_host_entry_argument_errors(lib):
    import ctypes as C
    lib.attn_fwd_host.argtypes = [C.c_void_p] * 5 + [C.c_int] * 6 + [C.c_float, C.c_int, C.c_void_p]
    b = Buf()
    p = b.p
    # sizes, flags, scale and pointers are checked on the host before any device work
    assert lib.attn_fwd_host(p, p, p, p, p, 1, 2, 1, 8, 8, 65, 0.125, 0, None) == -1
    assert lib.attn_fwd_host(p, p, p, p, p, 1, 3, 2, 8, 8, 64, 0.125, 0, None) == -1
    assert lib.attn_fwd_host(p, p, p, p, p, 1, 2, 1, 8, 8, 64, float("nan"), 0, None) == -1
    assert lib.attn_fwd_host(p, p, p, p, p, 1, 2, 1, 8, 8, 64, 0.125, 3, None) == -1
    assert lib.attn_fwd_host(None, p, p, p, p, 1, 2, 1, 8, 8, 64, 0.125, 0, None) == -1
    assert lib.attn_fwd_host(p, p, p, p, None, 1, 2, 1, 8, 8, 64, 0.125, 0, None) == -1
    # host buffers need no alignment: a misaligned pointer fails only on the device side, not here
    assert lib.attn_fwd_host(None, None, None, None, None, 0, 2, 1, 8, 8, 64, 0.125, 0, None) == 0


def test_set_debug_arguments(lib):
    lib.attn_set_debug.argtypes = [ctypes.c_int, ctypes.c_longlong]
    assert lib.attn_set_debug(8, 0) == -1
    assert lib.attn_set_debug(2 | 4, 0) == 0
    assert lib.attn_set_debug(2, 0) == 0
    assert lib.attn_set_debug(0, -5) == -1
    assert lib.attn_set_debug(1, 1000000) == 0
    assert lib.attn_set_debug(0, 0) == 0


def test_missing_library_fails_loudly(tmp_path):
    code = ("import exact_attention_attn_gb300 as A\n"
            "try:\n    A.attn_version()\nexcept ImportError as e:\n    print('RAISED', e)\n")
    env = dict(os.environ, ATTN_GB300_LIB=str(tmp_path / "nope.so"), PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)
    assert "RAISED" in r.stdout and "no fallback" in r.stdout


def test_plain_c_client(lib, tmp_path):
    # the C ABI from plain C: header + shared library, no C++ and no torch
    import shutil
    import torch
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(lib._name)
    exe = str(tmp_path / "attn_client")
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_client", "attn_client.c"), "-L", libdir, "-lattn_gb300",
                        f"-Wl,-rpath,{libdir}", "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    args = [] if torch.cuda.is_available() else ["--no-device"]
    r = subprocess.run([exe] + args, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout + r.stderr


def test_masked_entry_argument_errors(lib):
    import ctypes as C
    lib.attn_fwd_masked.argtypes = ([C.c_void_p] * 4 + [C.c_longlong] * 3 + [C.c_void_p] * 2 + [C.c_int] * 6 +
                                    [C.c_float, C.c_int, C.c_void_p])
    b = Buf()
    p = b.p
    ARG, ALIGN = -1, -2

    def masked(mask, sb=0, sh=0, sq=8, D=64, causal=0, B=1):
        return lib.attn_fwd_masked(p, p, p, mask, sb, sh, sq, p, p, B, 2, 1, 8, 8, D, 0.125, causal, None)

    assert masked(None) == ARG                 # a mask is required
    assert masked(p, sq=-8) == ARG             # negative stride
    assert masked(p, sb=-16) == ARG
    assert masked(p, sq=12) == ALIGN           # not a multiple of 8 elements
    assert masked(p, sh=4) == ALIGN
    assert masked(p + 2) == ALIGN              # misaligned base
    assert masked(p, D=96) == ARG              # the size checks of attn_fwd
    assert masked(p, causal=3) == ARG
    assert masked(p, B=0) == 0                 # empty problem: nothing to do


def test_backward_entry_argument_errors(lib):
    import ctypes as C
    lib.attn_bwd.argtypes = [C.c_void_p] * 9 + [C.c_int] * 6 + [C.c_float, C.c_int, C.c_void_p]
    b = Buf()
    p = b.p
    ARG, ALIGN = -1, -2

    def bwd(D=64, ptrs=None, causal=0, B=1, Nq=8, Nkv=8, scale=0.125):
        ptrs = ptrs or [p] * 9
        return lib.attn_bwd(*ptrs, B, 2, 1, Nq, Nkv, D, scale, causal, None)

    assert bwd(D=256) == ARG                   # head dims 64 and 128 only
    assert bwd(D=96) == ARG
    assert bwd(causal=2) == ARG
    assert bwd(scale=float("nan")) == ARG
    assert bwd(ptrs=[p] * 5 + [None] + [p] * 3) == ARG   # no lse
    assert bwd(ptrs=[p] * 8 + [None]) == ARG              # no dv
    assert bwd(ptrs=[p + 4] + [p] * 8) == ALIGN
    assert bwd(ptrs=[p] * 6 + [p + 8] + [p] * 2) == ALIGN
    assert bwd(B=0, ptrs=[None] * 9) == 0                # empty problem


def test_fp8_entry_argument_errors(lib):
    import ctypes as C
    lib.attn_fp8_quantize.argtypes = [C.c_void_p] * 9 + [C.c_int] * 6 + [C.c_void_p]
    lib.attn_fwd_fp8.argtypes = [C.c_void_p] * 8 + [C.c_int] * 6 + [C.c_float, C.c_int, C.c_void_p]
    b = Buf()
    p = b.p
    ARG, ALIGN = -1, -2
    assert lib.attn_fp8_quantize(*([p] * 9), 1, 2, 1, 8, 8, 64, None) == ARG    # head dim 128 only
    assert lib.attn_fp8_quantize(*([p] * 8), None, 1, 2, 1, 8, 8, 128, None) == ARG
    assert lib.attn_fp8_quantize(p + 4, *([p] * 8), 1, 2, 1, 8, 8, 128, None) == ALIGN
    assert lib.attn_fwd_fp8(*([p] * 8), 1, 2, 1, 8, 8, 128, 0.0, 0, None) == ARG   # scale must be > 0
    assert lib.attn_fwd_fp8(*([p] * 8), 1, 2, 1, 8, 8, 128, float("nan"), 0, None) == ARG
    assert lib.attn_fwd_fp8(*([p] * 8), 1, 2, 1, 8, 8, 128, 0.1, 2, None) == ARG
    assert lib.attn_fwd_fp8(*([p] * 8), 1, 2, 1, 8, 8, 256, 0.1, 0, None) == ARG
    assert lib.attn_fwd_fp8(*([None] * 8), 0, 2, 1, 8, 8, 128, 0.1, 0, None) == 0
