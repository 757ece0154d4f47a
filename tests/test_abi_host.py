"""C ABI checks that need no GPU: the libraries build for sm_103a, export
every function the headers declare, and reject bad arguments on the host
before any CUDA call."""
import ctypes as C
import os
import re

import pytest

import oracle
import sub_bit_weight_binary_b300 as sb
from sub_bit_weight_binary_b300 import build as sbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libs():
    paths = sbuild.build()
    return {os.path.basename(p): C.CDLL(p) for p in paths}


def declared(header):
    text = open(os.path.join(ROOT, "include", header), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bonsai_\w+)\s*\(", text)))


def test_headers_declare_the_boundary():
    names = declared("bonsai.h")
    for f in ("bonsai_packed_row_bytes", "bonsai_pack_binary", "bonsai_pack_ternary",
              "bonsai_gemv", "bonsai_gemm", "bonsai_xnor_gemm", "bonsai_binarize_activations",
              "bonsai_gemm_swiglu", "bonsai_hadamard", "bonsai_gemv_host", "bonsai_selftest_wait_timeout",
              "bonsai_check_async",
              "bonsai_status_string"):
        assert f in names


@pytest.mark.parametrize("header,lib", [("bonsai.h", "libbonsai.so"),
                                        ("bonsai_synth.h", "libbonsai_synth.so")])
def test_every_declared_symbol_is_exported(libs, header, lib):
    L = libs[lib]
    for name in declared(header):
        assert hasattr(L, name), "%s does not export %s" % (lib, name)


def test_weights_struct_layout_matches_the_header(tmp_path):
    """The binding's ctypes struct has the field offsets and size that a C
    compiler gives bonsai_weights from include/bonsai.h (flags last)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in sb.bonsai_weights_t._fields_]
    assert fields == ["format", "n", "k", "row_bytes", "packed", "scales", "flags"]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"bonsai.h\"\n"
                   "int main(void) { printf(\"%zu" + " %zu" * len(fields) + "\\n\", "
                   "sizeof(bonsai_weights)" +
                   "".join(", offsetof(bonsai_weights, %s)" % f for f in fields) +
                   "); return 0; }\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [C.sizeof(sb.bonsai_weights_t)] + [getattr(sb.bonsai_weights_t, f).offset
                                              for f in fields]
    assert got == want


def test_built_for_sm103a():
    # the objects carry sm_103a code (cuobjdump is not used: only the
    # compiler's own record of the target in the build flags is checked)
    assert "arch=compute_103a,code=sm_103a" in " ".join(sbuild.ARCH)


def test_row_bytes_and_status_strings(libs, oracle_lib):
    for fmt in (1, 2):
        for k in (128, 256, 640, 1024, 5120, 17408):
            assert sb.bonsai_packed_row_bytes(fmt, k) == oracle.row_bytes(fmt, k)
        for bad in (0, -128, 100, 129):
            assert sb.bonsai_packed_row_bytes(fmt, bad) == -1
    assert sb.bonsai_packed_row_bytes(3, 128) == -1
    for code, name in sb.STATUS.items():
        assert sb.bonsai_status_string(code) == name
    assert sb.bonsai_status_string(99) == "BONSAI_ERR_UNKNOWN"


def W(fmt=1, n=16, k=256, row_bytes=None, packed=0x10000, scales=0x20000, flags=0):
    if row_bytes is None:
        row_bytes = sb.bonsai_packed_row_bytes(fmt, k)
    return sb.bonsai_weights_t(fmt, n, k, row_bytes, packed, scales, flags)


# Each case fails a host check, so nothing is launched and no pointer is read.
BAD_GEMV = [
    ("null packed", dict(packed=None), "BONSAI_ERR_INVALID_ARG"),
    ("null scales", dict(scales=None), "BONSAI_ERR_INVALID_ARG"),
    ("format", dict(fmt=3), "BONSAI_ERR_INVALID_ARG"),
    ("flags", dict(flags=4), "BONSAI_ERR_INVALID_ARG"),
    ("n=0", dict(n=0), "BONSAI_ERR_INVALID_ARG"),
    ("k%128", dict(k=200, row_bytes=32), "BONSAI_ERR_SHAPE"),
    ("short row", dict(row_bytes=16), "BONSAI_ERR_SHAPE"),
    ("row%16", dict(row_bytes=40), "BONSAI_ERR_SHAPE"),
    ("ter row%64", dict(fmt=2, row_bytes=80), "BONSAI_ERR_SHAPE"),
    ("ter short", dict(fmt=2, k=5120, row_bytes=960), "BONSAI_ERR_SHAPE"),
    ("align packed", dict(packed=0x10008), "BONSAI_ERR_ALIGN"),
    ("align scales", dict(scales=0x20002), "BONSAI_ERR_ALIGN"),
    ("huge k", dict(k=1 << 21, row_bytes=1 << 18), "BONSAI_ERR_UNSUPPORTED"),
]


@pytest.mark.parametrize("what,kw,expect", BAD_GEMV, ids=[c[0] for c in BAD_GEMV])
def test_gemv_host_checks(libs, what, kw, expect):
    L = sb.lib()
    w = W(**kw)
    st = L.bonsai_gemv(C.byref(w), 0x30000, 0x40000, None)
    assert sb.STATUS[st] == expect


def test_other_host_checks(libs):
    L = sb.lib()
    w = W()
    assert sb.STATUS[L.bonsai_gemv(None, 0x30000, 0x40000, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[L.bonsai_gemv(C.byref(w), None, 0x40000, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[L.bonsai_gemv(C.byref(w), 0x30004, 0x40000, None)] == "BONSAI_ERR_ALIGN"
    assert sb.STATUS[L.bonsai_gemm(C.byref(w), 0x30000, 0, 0x40000, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[L.bonsai_gemm(C.byref(w), 0x30000, 4, 0x40002, None)] == "BONSAI_ERR_ALIGN"
    wt = W(fmt=2)
    assert sb.STATUS[L.bonsai_xnor_gemm(0x50000, 0x60000, 4, C.byref(wt), 0x70000, None, None)] \
        == "BONSAI_ERR_FORMAT"
    assert sb.STATUS[L.bonsai_xnor_gemm(0x50000, 0x60000, 4, C.byref(w), None, None, None)] \
        == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[L.bonsai_xnor_gemm(0x50004, 0x60000, 4, C.byref(w), 0x70000, None, None)] \
        == "BONSAI_ERR_ALIGN"
    assert sb.STATUS[L.bonsai_gemm_swiglu(C.byref(w), None, 4, 0x40000, None)] \
        == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[L.bonsai_gemm_swiglu(C.byref(w), 0x30000, 4, 0x40008, None)] \
        == "BONSAI_ERR_ALIGN"
    w24 = W(n=24)
    assert sb.STATUS[L.bonsai_gemm_swiglu(C.byref(w24), 0x30000, 4, 0x40000, None)] \
        == "BONSAI_ERR_SHAPE"
    gh = L.bonsai_gemv_host
    assert sb.STATUS[gh(C.byref(w), None, 0x30000, 0x40000, 0x50000, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[gh(C.byref(w), 0x10000, 0x30008, 0x40000, 0x50000, None)] == "BONSAI_ERR_ALIGN"
    assert sb.STATUS[gh(C.byref(W(fmt=3)), 0x10000, 0x30000, 0x40000, 0x50000, None)] \
        == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[L.bonsai_selftest_wait_timeout(10, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[L.bonsai_selftest_wait_timeout(10 ** 9, None)] == "BONSAI_ERR_INVALID_ARG"
    hd = L.bonsai_hadamard
    assert sb.STATUS[hd(None, 2, 256, 128, None, 0x50000, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[hd(0x40000, 2, 256, 96, None, 0x50000, None)] == "BONSAI_ERR_UNSUPPORTED"
    assert sb.STATUS[hd(0x40000, 2, 256, 2048, None, 0x50000, None)] == "BONSAI_ERR_UNSUPPORTED"
    assert sb.STATUS[hd(0x40000, 2, 384, 256, None, 0x50000, None)] == "BONSAI_ERR_SHAPE"
    assert sb.STATUS[hd(0x40000, 2, 200, 8, None, 0x50000, None)] == "BONSAI_ERR_SHAPE"
    assert sb.STATUS[hd(0x40008, 2, 256, 128, None, 0x50000, None)] == "BONSAI_ERR_ALIGN"
    assert sb.STATUS[hd(0x40000, 2, 256, 128, 0x60002, 0x50000, None)] == "BONSAI_ERR_ALIGN"
    # overlapping but not identical buffers
    assert sb.STATUS[hd(0x40000, 2, 256, 128, None, 0x40100, None)] == "BONSAI_ERR_INVALID_ARG"
    bz = L.bonsai_binarize_activations
    assert sb.STATUS[bz(None, 4, 128, 0x50000, 0x60000, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[bz(0x40000, 0, 128, 0x50000, 0x60000, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[bz(0x40000, 4, 96, 0x50000, 0x60000, None)] == "BONSAI_ERR_SHAPE"
    assert sb.STATUS[bz(0x40000, 4, 1 << 21, 0x50000, 0x60000, None)] == "BONSAI_ERR_UNSUPPORTED"
    assert sb.STATUS[bz(0x40000, 4, 128, 0x50004, 0x60000, None)] == "BONSAI_ERR_ALIGN"
    assert sb.STATUS[bz(0x40000, 4, 128, 0x50000, 0x60002, None)] == "BONSAI_ERR_ALIGN"
    for f in (L.bonsai_pack_binary, L.bonsai_pack_ternary):
        assert sb.STATUS[f(None, 2, 128, 0x10000, 64, None)] == "BONSAI_ERR_INVALID_ARG"
        assert sb.STATUS[f(0x10000, -1, 128, 0x20000, 64, None)] == "BONSAI_ERR_INVALID_ARG"
        assert sb.STATUS[f(0x10000, 2, 100, 0x20000, 64, None)] == "BONSAI_ERR_SHAPE"
        assert sb.STATUS[f(0x10001, 2, 128, 0x20000, 64, None)] == "BONSAI_ERR_ALIGN"
    assert sb.STATUS[L.bonsai_pack_binary(0x10000, 2, 128, 0x20000, 8, None)] == "BONSAI_ERR_SHAPE"
    assert sb.STATUS[L.bonsai_pack_ternary(0x10000, 2, 128, 0x20000, 32, None)] == "BONSAI_ERR_SHAPE"
    # zero rows is a valid no-op (no launch)
    assert sb.STATUS[L.bonsai_pack_binary(0x10000, 0, 128, 0x20000, 16, None)] == "BONSAI_OK"


def test_plan_host_checks(libs):
    """Plan calls reject bad steps on the host before any CUDA call."""
    L = sb.lib()
    assert L.bonsai_decode_plan_bytes(0) == -1
    assert L.bonsai_decode_plan_bytes(5000) == -1
    nb = L.bonsai_decode_plan_bytes(3)
    assert nb > 0 and nb % 128 == 0

    def steps(fmt=2, after=(-1, 0, 1), swiglu=(0, 0, 0), x=0x30000, y=0x40000, n=32):
        arr = (sb.bonsai_decode_step_t * len(after))()
        for i, a in enumerate(after):
            arr[i].w = W(fmt=fmt, n=n)
            arr[i].x, arr[i].y, arr[i].swiglu, arr[i].after = x, y, swiglu[i], a
        return arr
    init, run = L.bonsai_decode_plan_init, L.bonsai_decode_run
    good = steps()
    assert sb.STATUS[init(good, 0, 0x80000, nb, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[init(good, 3, None, nb, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[init(good, 3, 0x80040, nb, None)] == "BONSAI_ERR_ALIGN"
    assert sb.STATUS[init(good, 3, 0x80000, nb - 128, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[init(steps(after=(-1, 1, 0)), 3, 0x80000, nb, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[init(steps(after=(-2, 0, 0)), 3, 0x80000, nb, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[init(steps(fmt=1), 3, 0x80000, nb, None)] == "BONSAI_ERR_FORMAT"
    assert sb.STATUS[init(steps(swiglu=(0, 2, 0)), 3, 0x80000, nb, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[init(steps(swiglu=(0, 1, 0), n=24), 3, 0x80000, nb, None)] == "BONSAI_ERR_SHAPE"
    assert sb.STATUS[init(steps(x=0x30004), 3, 0x80000, nb, None)] == "BONSAI_ERR_ALIGN"
    assert sb.STATUS[run(steps(after=(-1, 2, 1)), 3, 0x80000, None)] == "BONSAI_ERR_INVALID_ARG"
    assert sb.STATUS[run(good, 3, 0x80010, None)] == "BONSAI_ERR_ALIGN"
    assert sb.STATUS[L.bonsai_selftest_plan_wait(10, None)] == "BONSAI_ERR_INVALID_ARG"


def test_binding_refuses_cpu_tensors(libs):
    import torch
    w = sb.Weights(1, 4, 128, torch.zeros(4, 16, dtype=torch.uint8),
                   torch.zeros(4, 1, dtype=torch.float16))
    with pytest.raises(ValueError):
        sb.bonsai_gemv(w, torch.zeros(128, dtype=torch.float16),
                       torch.zeros(4, dtype=torch.float16), stream=0)


def test_interleave_gate_up_row_order():
    """interleave_gate_up puts gate row f at 16*(f//8) + f%8 and up row f
    8 rows below it, for numpy arrays and torch tensors."""
    import numpy as np
    import torch
    f = 24
    gate = np.arange(f * 3).reshape(f, 3)
    up = 1000 + np.arange(f * 3).reshape(f, 3)
    out = sb.interleave_gate_up(gate, up)
    for r in range(f):
        assert np.array_equal(out[16 * (r // 8) + r % 8], gate[r])
        assert np.array_equal(out[16 * (r // 8) + r % 8 + 8], up[r])
    tout = sb.interleave_gate_up(torch.from_numpy(gate), torch.from_numpy(up))
    assert np.array_equal(tout.numpy(), out)
    with pytest.raises(ValueError):
        sb.interleave_gate_up(gate[:12], up[:12])


def test_weights_struct_is_cached_and_rebuilt_on_assignment():
    import torch
    w = sb.Weights(1, 4, 128, torch.zeros(4, 16, dtype=torch.uint8),
                   torch.zeros(4, 1, dtype=torch.float16))
    w.__dict__["_cs"] = "cached"           # stands for a built struct
    assert w.c_struct() == "cached"
    w.flags = 1                            # any assignment drops it
    assert "_cs" not in w.__dict__
