"""ctypes binding of libbonsai_synth.so, the GPU twin of synth.py.

Fills device tensors with the same seeded values synth.py draws on the host
(integer codes, raw bits, uniform FP16 scales). Input generation only.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbonsai_synth.so")

_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libbonsai_synth.so is not built: run "
                              "python -m sub_bit_weight_binary_b300.build")
        L = C.CDLL(LIB_PATH)
        U64, I64, P = C.c_uint64, C.c_int64, C.c_void_p
        for name in ("bonsai_synth_bits32", "bonsai_synth_ternary_codes",
                     "bonsai_synth_binary_codes"):
            f = getattr(L, name)
            f.argtypes = [U64, U64, I64, I64, P, P]
            f.restype = C.c_int
        L.bonsai_synth_uniform_f16.argtypes = [U64, U64, I64, I64, C.c_double, C.c_double, P, P]
        L.bonsai_synth_uniform_f16.restype = C.c_int
        _lib = L
    return _lib


def _s(stream):
    import torch
    return torch.cuda.current_stream().cuda_stream if stream is None else stream.cuda_stream


def _chk(rc, what):
    if rc != 0:
        raise RuntimeError("%s failed with %d" % (what, rc))


def bits32(seed, tid, start, out, stream=None):
    """out: int32 CUDA tensor; filled with r(start + j) >> 32."""
    _chk(lib().bonsai_synth_bits32(seed, tid, start, out.numel(), out.data_ptr(), _s(stream)),
         "bonsai_synth_bits32")


def ternary_codes(seed, tid, start, out, stream=None):
    _chk(lib().bonsai_synth_ternary_codes(seed, tid, start, out.numel(), out.data_ptr(),
                                          _s(stream)), "bonsai_synth_ternary_codes")


def binary_codes(seed, tid, start, out, stream=None):
    _chk(lib().bonsai_synth_binary_codes(seed, tid, start, out.numel(), out.data_ptr(),
                                         _s(stream)), "bonsai_synth_binary_codes")


def uniform_f16(seed, tid, start, lo, hi, out, stream=None):
    """out: float16 CUDA tensor."""
    _chk(lib().bonsai_synth_uniform_f16(seed, tid, start, out.numel(), lo, hi, out.data_ptr(),
                                        _s(stream)), "bonsai_synth_uniform_f16")
