"""Python face of the plain-C oracle (oracle.c).

TEST INFRASTRUCTURE. Only tests/, the package's smoke() check and the
benchmark's CPU-baseline leg may import this module. The CUDA path never
imports it, and it never imports the CUDA path.

Arrays are numpy; FP16 values travel as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

FMT_BINARY = 1
FMT_TERNARY = 2
OK = 0
ERR_BAD_CODE = 8
GROUP = 128


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with the host C compiler."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


_lib = None


def configure(L):
    """Declare the C signatures on a loaded oracle library."""
    P = C.c_void_p
    I64 = C.c_int64
    L.oracle_half_to_double.argtypes = [C.c_uint16]
    L.oracle_half_to_double.restype = C.c_double
    L.oracle_row_bytes.argtypes = [C.c_int, I64]
    L.oracle_row_bytes.restype = I64
    for name in ("oracle_pack_binary", "oracle_pack_ternary"):
        f = getattr(L, name)
        f.argtypes = [P, I64, I64, P, I64]
        f.restype = C.c_int
    for name in ("oracle_unpack_binary", "oracle_unpack_ternary"):
        f = getattr(L, name)
        f.argtypes = [P, I64, I64, I64, P]
        f.restype = C.c_int
    L.oracle_linear.argtypes = [C.c_int, P, I64, P, I64, I64, P, I64,
                                P, I64, P, I64, P, P]
    L.oracle_linear.restype = C.c_int
    L.oracle_swiglu.argtypes = [C.c_int, P, I64, P, I64, I64, P, I64, P, I64, P, I64,
                                P, P, P, P, P]
    L.oracle_swiglu.restype = C.c_int
    L.oracle_hadamard.argtypes = [P, I64, I64, I64, P, P]
    L.oracle_hadamard.restype = C.c_int
    L.oracle_binarize.argtypes = [P, I64, I64, P, P]
    L.oracle_binarize.restype = C.c_int
    L.oracle_xnor.argtypes = [P, P, I64, P, I64, P, I64, I64,
                              P, I64, P, I64, P, P, P]
    L.oracle_xnor.restype = C.c_int
    L.oracle_compare_f16.argtypes = [P, P, P, I64, C.c_double, P, P]
    L.oracle_compare_f16.restype = I64
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = configure(C.CDLL(LIB))
    return _lib


def use_library(L):
    """Swap the loaded library (tests load deliberately broken copies of
    oracle.c to check that the pins catch them). Returns the previous one."""
    global _lib
    prev = _lib
    _lib = L
    return prev


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed with oracle status %d" % (what, status))
        self.status = status


def _check(st: int, what: str):
    if st != OK:
        raise OracleError(st, what)


def half_to_double(h: int) -> float:
    return lib().oracle_half_to_double(int(h))


def row_bytes(fmt: int, k: int) -> int:
    return int(lib().oracle_row_bytes(fmt, k))


def pack_binary(codes: np.ndarray, row_bytes_: int | None = None) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    rows, k = codes.shape
    rb = row_bytes(FMT_BINARY, k) if row_bytes_ is None else row_bytes_
    out = np.empty((rows, rb), dtype=np.uint8)
    _check(lib().oracle_pack_binary(_p(codes), rows, k, _p(out), rb), "pack_binary")
    return out


def unpack_binary(packed: np.ndarray, k: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed).view(np.uint8)
    rows, rb = packed.shape
    out = np.empty((rows, k), dtype=np.int8)
    _check(lib().oracle_unpack_binary(_p(packed), rows, k, rb, _p(out)), "unpack_binary")
    return out


def pack_ternary(codes: np.ndarray, row_bytes_: int | None = None) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    rows, k = codes.shape
    rb = row_bytes(FMT_TERNARY, k) if row_bytes_ is None else row_bytes_
    out = np.empty((rows, rb), dtype=np.uint8)
    _check(lib().oracle_pack_ternary(_p(codes), rows, k, _p(out), rb), "pack_ternary")
    return out


def unpack_ternary(packed: np.ndarray, k: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    rows, rb = packed.shape
    out = np.empty((rows, k), dtype=np.int8)
    _check(lib().oracle_unpack_ternary(_p(packed), rows, k, rb, _p(out)), "unpack_ternary")
    return out


def linear(fmt: int, packed: np.ndarray, scales: np.ndarray, x: np.ndarray,
           n_sel=None, m_sel=None):
    """(y, norm), each float64 [len(m_sel)][len(n_sel)].

    packed: uint8 [n][row_bytes] (any dtype viewed as bytes per row);
    scales: uint16 [n][k/128]; x: uint16 [m][k]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    m, k = x.shape
    packed = np.ascontiguousarray(packed)
    n = packed.shape[0]
    packed = packed.view(np.uint8).reshape(n, -1)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    n_sel = np.arange(n, dtype=np.int64) if n_sel is None else np.ascontiguousarray(n_sel, dtype=np.int64)
    m_sel = np.arange(m, dtype=np.int64) if m_sel is None else np.ascontiguousarray(m_sel, dtype=np.int64)
    y = np.empty((len(m_sel), len(n_sel)), dtype=np.float64)
    nrm = np.empty_like(y)
    _check(lib().oracle_linear(fmt, _p(packed), packed.shape[1], _p(scales), n, k,
                               _p(x), m, _p(n_sel), len(n_sel), _p(m_sel), len(m_sel),
                               _p(y), _p(nrm)), "linear")
    return y, nrm


def xnor(a_bits: np.ndarray, a_scale: np.ndarray, w_packed: np.ndarray,
         scales: np.ndarray, k: int, n_sel=None, m_sel=None):
    """(d int64, y float64, norm float64), each [len(m_sel)][len(n_sel)]."""
    a_bits = np.ascontiguousarray(a_bits)
    m = a_bits.shape[0]
    a_bytes = a_bits.view(np.uint8).reshape(m, -1)
    a_scale = np.ascontiguousarray(a_scale, dtype=np.uint16)
    w_packed = np.ascontiguousarray(w_packed)
    n = w_packed.shape[0]
    w_bytes = w_packed.view(np.uint8).reshape(n, -1)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    n_sel = np.arange(n, dtype=np.int64) if n_sel is None else np.ascontiguousarray(n_sel, dtype=np.int64)
    m_sel = np.arange(m, dtype=np.int64) if m_sel is None else np.ascontiguousarray(m_sel, dtype=np.int64)
    d = np.empty((len(m_sel), len(n_sel)), dtype=np.int64)
    y = np.empty(d.shape, dtype=np.float64)
    nrm = np.empty(d.shape, dtype=np.float64)
    _check(lib().oracle_xnor(_p(a_bytes), _p(a_scale), m, _p(w_bytes), w_bytes.shape[1],
                             _p(scales), n, k, _p(n_sel), len(n_sel), _p(m_sel), len(m_sel),
                             _p(d), _p(y), _p(nrm)), "xnor")
    return d, y, nrm


def swiglu(fmt: int, packed: np.ndarray, scales: np.ndarray, x: np.ndarray,
           f_sel=None, m_sel=None):
    """Gated feed-forward input h = silu(g) * u of the interleaved gate/up
    matrix packed [2F][row_bytes] (16-row blocks: 8 gate rows, then the 8 up
    rows of the same features). Returns (h, g, u, norm_g, norm_u), each
    [len(m_sel)][len(f_sel)] float64."""
    packed = np.ascontiguousarray(packed)
    n = packed.shape[0]
    pb = packed.view(np.uint8).reshape(n, -1)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    m, k = x.shape
    f_sel = np.arange(n // 2, dtype=np.int64) if f_sel is None else np.ascontiguousarray(f_sel, dtype=np.int64)
    m_sel = np.arange(m, dtype=np.int64) if m_sel is None else np.ascontiguousarray(m_sel, dtype=np.int64)
    outs = [np.empty((len(m_sel), len(f_sel)), dtype=np.float64) for _ in range(5)]
    _check(lib().oracle_swiglu(fmt, _p(pb), pb.shape[1], _p(scales), n, k, _p(x), m,
                               _p(f_sel), len(f_sel), _p(m_sel), len(m_sel),
                               *[_p(o) for o in outs]), "swiglu")
    return tuple(outs)


def hadamard(x: np.ndarray, block: int, sign_bits=None):
    """Block-diagonal signed Hadamard rotation of FP16 rows x [m][k]
    (float64 [m][k]); sign_bits: uint32 [k/32] (bit 1 = +1) or None."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    m, k = x.shape
    out = np.empty((m, k), dtype=np.float64)
    sb = None if sign_bits is None else np.ascontiguousarray(sign_bits, dtype=np.uint32)
    _check(lib().oracle_hadamard(_p(x), m, k, block, None if sb is None else _p(sb), _p(out)),
           "hadamard")
    return out


def binarize(x: np.ndarray):
    """(bits uint32 [m][k/32], a_scale float64 [m]) of FP16 rows x [m][k]:
    bit 1 where x >= 0, a_scale = mean |x| per row."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    m, k = x.shape
    bits = np.zeros((m, k // 32), dtype=np.uint32)
    a_s = np.empty(m, dtype=np.float64)
    _check(lib().oracle_binarize(_p(x), m, k, _p(bits), _p(a_s)), "binarize")
    return bits, a_s


def compare_f16(y_gpu: np.ndarray, y_ref: np.ndarray, norm: np.ndarray,
                tol: float = 2e-3):
    """(failures, first_bad_index, worst |err|/norm) of the acceptance rule."""
    y_gpu = np.ascontiguousarray(y_gpu, dtype=np.uint16).ravel()
    y_ref = np.ascontiguousarray(y_ref, dtype=np.float64).ravel()
    norm = np.ascontiguousarray(norm, dtype=np.float64).ravel()
    assert y_gpu.size == y_ref.size == norm.size
    first = np.zeros(1, dtype=np.int64)
    worst = np.zeros(1, dtype=np.float64)
    bad = lib().oracle_compare_f16(_p(y_gpu), _p(y_ref), _p(norm), y_gpu.size, tol,
                                   _p(first), _p(worst))
    return int(bad), int(first[0]), float(worst[0])
