"""Shared helpers of the GPU parity tests: seeded inputs on both sides, the
oracle's reference, and guard bands around every output buffer."""
from __future__ import annotations

import numpy as np

import oracle
import sub_bit_weight_binary_b300 as sb
from sub_bit_weight_binary_b300 import synth

TOL = 2e-3          # |y - y_ref| <= TOL * sum|x*s*w| per output
GUARD = 512         # guard elements after each output buffer
GUARD_F16 = 0x7E5A  # a NaN pattern no kernel writes


def torch():
    import torch as t
    return t


def dev(a: np.ndarray):
    """numpy -> CUDA tensor (uint16 arrays become float16 bit-for-bit)."""
    t = torch()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.float16)
    return t.from_numpy(a).cuda()


def host(t) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    return a


class Guarded:
    """A CUDA buffer of `shape` followed by GUARD elements of a fixed
    pattern; .check() asserts that no kernel wrote past the end."""

    def __init__(self, shape, dtype, fill=None):
        t = torch()
        n = int(np.prod(shape))
        self.full = t.empty(n + GUARD, dtype=dtype, device="cuda")
        if dtype == t.float16:
            self.full.view(t.int16).fill_(GUARD_F16)
            self.pattern = GUARD_F16
        elif dtype == t.int32:
            self.full.fill_(0x5A5A5A5A)
            self.pattern = 0x5A5A5A5A
        else:
            self.full.fill_(0xA5)
            self.pattern = 0xA5
        self.t = self.full[:n].view(*shape)
        if fill is not None:
            self.t.copy_(fill)

    def check(self):
        tail = host(self.full[-GUARD:])
        assert np.all(tail == np.array(self.pattern).astype(tail.dtype)), "write past the end"


def binary_weights(seed, n, k, flags=0):
    """(Weights on device, packed bytes on host, scales on host)."""
    words = synth.gen_binary_words(seed, n, k)
    packed = words.view(np.uint8).reshape(n, -1)
    scales = synth.gen_scales(seed, n, k)
    w = sb.Weights(sb.BONSAI_FMT_BINARY, n, k, dev(packed), dev(scales), flags)
    return w, packed, scales


def ternary_weights(seed, n, k, flags=0):
    """Codes drawn on the host; the GPU side packs them with bonsai_pack_ternary,
    the oracle side with its own packer (the pack tests compare the two)."""
    t = torch()
    codes = synth.gen_ternary_codes(seed, n, k)
    rb = sb.bonsai_packed_row_bytes(sb.BONSAI_FMT_TERNARY, k)
    packed_gpu = t.empty((n, rb), dtype=t.uint8, device="cuda")
    sb.bonsai_pack_ternary(dev(codes), packed_gpu)
    packed = oracle.pack_ternary(codes)
    scales = synth.gen_scales(seed, n, k)
    w = sb.Weights(sb.BONSAI_FMT_TERNARY, n, k, packed_gpu, dev(scales), flags)
    return w, packed, scales


def weights(fmt, seed, n, k, flags=0):
    return binary_weights(seed, n, k, flags) if fmt == sb.BONSAI_FMT_BINARY \
        else ternary_weights(seed, n, k, flags)


def assert_close(y_gpu_u16, y_ref, norm, what=""):
    bad, first, worst = oracle.compare_f16(y_gpu_u16, y_ref, norm, TOL)
    assert bad == 0, "%s: %d outputs outside %g*norm (first flat index %d, worst %.3g)" % (
        what, bad, TOL, first, worst)
    return worst


def assert_swiglu_close(h_gpu_u16, h, g, u, norm_g, norm_u, what=""):
    """h = silu(g) * u from g and u that each carry the products' error
    (<= TOL * norm). |silu'| <= 1.1 and |silu(g)| <= |g| give
        |dh| <= 1.1 * Eg * (|u| + Eu) + |g| * Eu,   E* = TOL * norm_*,
    and the single FP16 rounding of h adds 2^-11 of |h| + that (2^-10 kept).
    A zero bound (no gate or no up weights) requires h = +-0 exactly."""
    eg, eu = TOL * norm_g, TOL * norm_u
    b = 1.1 * eg * (np.abs(u) + eu) + np.abs(g) * eu
    b = b + 2.0 ** -10 * (np.abs(h) + b)
    bad, first, worst = oracle.compare_f16(h_gpu_u16, h, b, 1.0)
    assert bad == 0, "%s: %d outputs outside the bound (first flat index %d, worst %.3g)" % (
        what, bad, first, worst)
    return worst
