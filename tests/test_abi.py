"""The C ABI library: it builds for sm_103a, loads, exports every symbol that
include/kda.h declares, and rejects bad arguments on the host (status codes,
nothing launched).  No test here needs a GPU or touches device memory."""
import ctypes
import os
import re
import subprocess

import pytest

from gated_delta_rule_26_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:[A-Za-z_]\w*[\s*]+)+(kda_\w+)\s*\(", text,
                                 flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    path = kbuild.build()
    return ctypes.CDLL(path)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for core in ("kda_gate", "kda_chunk_forward", "kda_recurrent_step", "kda_status_string",
                 "kda_launch_count"):
        assert core in names, core


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", kbuild.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name


def test_status_strings(lib):
    lib.kda_status_string.restype = ctypes.c_char_p
    assert lib.kda_status_string(0) == b"ok"
    assert lib.kda_status_string(-3) == b"pointer not 16-byte aligned"
    assert lib.kda_status_string(12345) == b"unknown status"


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int)]


def _fwd(lib, dims, chunk=64, dtype=1, misalign=0, null_q=False, fn="kda_chunk_forward"):
    p = 1 << 20  # fake, never dereferenced: every call below is rejected on the host
    vp = ctypes.c_void_p
    f = getattr(lib, fn)
    f.argtypes = [ctypes.c_void_p, ctypes.c_int] + [vp] * 7 + \
        [ctypes.c_float, vp, ctypes.c_int, vp, vp, vp]
    q = None if null_q else vp(p + misalign)
    return f(ctypes.byref(dims) if dims is not None else None, dtype, q,
             vp(p), vp(p), vp(p), vp(p), vp(p), vp(p), 0.1, None, chunk, vp(p), None, None)


def test_host_validation_rejects_bad_arguments(lib):
    assert _fwd(lib, None) == -1                              # null dims
    assert _fwd(lib, Dims(1, 1, 8, 128, 128), dtype=7) == -1  # bad dtype enum
    assert _fwd(lib, Dims(0, 1, 8, 128, 128)) == -1           # B < 1
    assert _fwd(lib, Dims(1, 1, -1, 128, 128)) == -1          # T < 0
    assert _fwd(lib, Dims(1, 1, 8, 7, 128)) == -2             # K not a multiple of 8
    assert _fwd(lib, Dims(1, 1, 8, 136, 128)) == -2           # K > 128
    assert _fwd(lib, Dims(1, 1, 8, 128, 256)) == -2           # V > 128
    assert _fwd(lib, Dims(1, 1, 8, 128, 128), chunk=48) == -2 # chunk not in {16, 32, 64}
    assert _fwd(lib, Dims(1, 1, 8, 128, 128), misalign=2) == -3
    assert _fwd(lib, Dims(1, 1, 8, 128, 128), null_q=True) == -1


@pytest.mark.parametrize("fn", ["kda_chunk_forward_split", "kda_chunk_forward_fused",
                                "kda_chunk_forward_scan"])
def test_tensor_core_forms_reject_other_shapes(lib, fn):
    # each form exists for bf16, K = V = 128, chunk 64 and T >= 1 only; everything else is
    # refused on the host (nothing is launched, so fake pointers are fine)
    assert _fwd(lib, Dims(1, 1, 64, 128, 128), dtype=0, fn=fn) == -2  # fp32 I/O
    assert _fwd(lib, Dims(1, 1, 64, 64, 128), fn=fn) == -2            # K = 64
    assert _fwd(lib, Dims(1, 1, 64, 128, 64), fn=fn) == -2            # V = 64
    assert _fwd(lib, Dims(1, 1, 64, 128, 128), chunk=32, fn=fn) == -2 # chunk 32
    assert _fwd(lib, Dims(1, 1, 0, 128, 128), fn=fn) == -2            # T = 0
    assert _fwd(lib, Dims(1, 1, 64, 128, 128), misalign=2, fn=fn) == -3
    assert _fwd(lib, None, fn=fn) == -1


def test_recurrent_step_requires_one_token(lib):
    vp = ctypes.c_void_p
    p = vp(1 << 20)
    lib.kda_recurrent_step.argtypes = [ctypes.c_void_p, ctypes.c_int] + [vp] * 7 + \
        [ctypes.c_float, vp, vp, vp]
    assert lib.kda_recurrent_step(ctypes.byref(Dims(2, 2, 2, 64, 64)), 1, p, p, p, p, p, p, p,
                                  0.1, p, p, None) == -1
    assert lib.kda_recurrent_step(ctypes.byref(Dims(2, 2, 1, 64, 64)), 1, p, p, p, p, p, p, p,
                                  0.1, vp((1 << 20) + 8), p, None) == -3   # state
    assert lib.kda_recurrent_step(ctypes.byref(Dims(2, 2, 1, 64, 64)), 1, vp((1 << 20) + 1), p,
                                  p, p, p, p, p, 0.1, p, p, None) == -3   # odd bf16 address


def test_gate_rejects_bad_chunk(lib):
    vp = ctypes.c_void_p
    p = vp(1 << 20)
    lib.kda_gate.argtypes = [ctypes.c_void_p, ctypes.c_int, vp, vp, vp, ctypes.c_int, vp, vp]
    assert lib.kda_gate(ctypes.byref(Dims(1, 1, 8, 64, 0)), 0, p, p, p, 24, p, None) == -2
    assert lib.kda_gate(ctypes.byref(Dims(1, 1, 8, 64, 0)), 0, None, p, p, 0, p, None) == -1


def _bwd(lib, dims, dtype=1, misalign=0, null_do=False, null_dq=False):
    p = 1 << 20  # fake, never dereferenced: every call below is rejected on the host
    vp = ctypes.c_void_p
    f = lib.kda_chunk_backward
    f.argtypes = [ctypes.c_void_p, ctypes.c_int] + [vp] * 7 + [ctypes.c_float] + [vp] * 12
    d_o = None if null_do else vp(p + misalign)
    dq = None if null_dq else vp(p)
    return f(ctypes.byref(dims) if dims is not None else None, dtype,
             vp(p), vp(p), vp(p), vp(p), vp(p), vp(p), vp(p), 0.1, None, d_o, None,
             dq, vp(p), vp(p), vp(p), vp(p), vp(p), vp(p), None, None)


def test_backward_rejects_bad_arguments(lib):
    assert _bwd(lib, None) == -1
    assert _bwd(lib, Dims(1, 1, 8, 128, 128), dtype=3) == -1
    assert _bwd(lib, Dims(1, 0, 8, 128, 128)) == -1
    assert _bwd(lib, Dims(1, 1, 8, 12, 128)) == -2
    assert _bwd(lib, Dims(1, 1, 8, 128, 256)) == -2
    assert _bwd(lib, Dims(1, 1, 8, 128, 128), misalign=4) == -3
    assert _bwd(lib, Dims(1, 1, 8, 128, 128), null_do=True) == -1
    assert _bwd(lib, Dims(1, 1, 8, 128, 128), null_dq=True) == -1


def test_header_is_plain_c_and_links_against_the_library(tmp_path):
    """include/kda.h compiles as C99 (no C++ or CUDA types in the signatures), and a C program
    that takes the address of every declared entry point links against libkda."""
    names = declared_functions()
    src = tmp_path / "use_kda.c"
    body = "\n".join(f"    (void)&{n};" for n in names)
    src.write_text('#include "kda.h"\nint main(void) {\n' + body + "\n    return 0;\n}\n")
    exe = tmp_path / "use_kda"
    lib_dir = os.path.dirname(kbuild.build())
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", lib_dir, "-lkda"], check=True)
