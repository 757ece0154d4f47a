"""Seeded synthetic inputs, host side.

A counter-based generator: element i of tensor `tid` under `seed` is

    key  = splitmix64(seed XOR (tid << 40))
    r(i) = splitmix64(key + i)            (64-bit wrap-around)

with splitmix64 as published by S. Vigna (add the golden-ratio increment
0x9E3779B97F4A7C15, then two xor-shift-multiply rounds with 0xBF58476D1CE4E5B9
and 0x94D049BB133111EB, then a final xor-shift by 31). Every element is a pure
function of (seed, tid, i), so any slice of a tensor can be regenerated alone
and the device twin (csrc/synth.cu) produces bit-identical integer tensors.

This module only draws inputs. It holds none of the products' arithmetic and
is shared by the oracle-side tests and the CUDA path.

Distributions (the workloads' value recipe):
  x          N(0,1) by Box-Muller in float64 from r(2i), r(2i+1), rounded to FP16
  scales     U[lo, hi) in float64, rounded to FP16 (lo, hi = 0.01, 0.05)
  bin words  raw bits: the high 32 bits of r(i) (Bernoulli(0.5) signs)
  bin codes  +1 if the top bit of r(i) is 1 else -1
  ter codes  t = r(i) >> 40 (24 bits): t < 5033165 -> -1, t < 11744051 -> 0,
             else +1, i.e. P(-1) = P(+1) = 0.3 and P(0) = 0.4
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)

# 24-bit thresholds of the ternary code distribution (0.3 and 0.7 of 2**24).
TER_T1 = 5033165
TER_T2 = 11744051

# Tensor ids, one per role. Sweep matrices use SWEEP_BASE + 16*layer + j.
TID_X = 1
TID_SCALES = 2
TID_WBIN = 3
TID_WTER = 4
TID_A_BITS = 5
TID_A_SCALE = 6
TID_CODES = 7
SWEEP_BASE = 0x100

SEED_BASE = 0xB0A5A1


def config_seed(config_id: int) -> int:
    """Seed of workload `config_id` (1-based)."""
    return SEED_BASE + int(config_id)


def splitmix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int) -> np.uint64:
    s = (int(seed) ^ (int(tid) << 40)) & 0xFFFFFFFFFFFFFFFF
    return splitmix64(np.array([s], dtype=np.uint64))[0]


def words(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    """r(start .. start+count-1) as uint64."""
    key = stream_key(seed, tid)
    idx = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return splitmix64(idx + key)


def bits32(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    """Raw random 32-bit words (the high half of r(i))."""
    return (words(seed, tid, start, count) >> np.uint64(32)).astype(np.uint32)


def binary_codes(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    w = words(seed, tid, start, count)
    return np.where((w >> np.uint64(63)) == 1, 1, -1).astype(np.int8)


def ternary_codes(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    t = words(seed, tid, start, count) >> np.uint64(40)
    out = np.ones(count, dtype=np.int8)  # +1
    out[t < TER_T2] = 0
    out[t < TER_T1] = -1
    return out


def uniform_f16(seed: int, tid: int, start: int, count: int,
                lo: float, hi: float) -> np.ndarray:
    """U[lo, hi) rounded to FP16; returned as uint16 bit patterns.

    u = (r >> 11) * 2**-53 exactly; v = lo + u * (hi - lo) with two float64
    roundings (multiply, then add); FP16 by round-to-nearest-even.
    """
    u = (words(seed, tid, start, count) >> np.uint64(11)).astype(np.float64)
    u = u * (2.0 ** -53)
    v = lo + u * (hi - lo)
    return v.astype(np.float16).view(np.uint16)


def normal_f16(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    """N(0,1) by Box-Muller, rounded to FP16; uint16 bit patterns."""
    w = words(seed, tid, 2 * start, 2 * count)
    u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return z.astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------------------
# Whole tensors of the workloads.

def gen_x(seed: int, m: int, k: int) -> np.ndarray:
    return normal_f16(seed, TID_X, 0, m * k).reshape(m, k)


def gen_scales(seed: int, n: int, k: int, tid: int = TID_SCALES,
               lo: float = 0.01, hi: float = 0.05) -> np.ndarray:
    g = k // 128
    return uniform_f16(seed, tid, 0, n * g, lo, hi).reshape(n, g)


def gen_binary_words(seed: int, n: int, k: int, tid: int = TID_WBIN,
                     row0: int = 0) -> np.ndarray:
    """Packed binary weights (rows row0 .. row0+n-1), uint32 [n][k/32]."""
    wpr = k // 32
    return bits32(seed, tid, row0 * wpr, n * wpr).reshape(n, wpr)


def gen_ternary_codes(seed: int, n: int, k: int, tid: int = TID_WTER,
                      row0: int = 0) -> np.ndarray:
    """int8 codes in {-1,0,+1}, [n][k] (rows row0 .. row0+n-1)."""
    return ternary_codes(seed, tid, row0 * k, n * k).reshape(n, k)


def gen_binary_codes(seed: int, n: int, k: int, tid: int = TID_CODES,
                     row0: int = 0) -> np.ndarray:
    return binary_codes(seed, tid, row0 * k, n * k).reshape(n, k)


def gen_xnor_inputs(seed: int, m: int, n: int, k: int):
    """(a_bits [m][k/32] u32, a_scale [m] fp16 bits, w_bits [n][k/32] u32,
    scales [n][k/128] fp16 bits) for the XNOR product."""
    a_bits = bits32(seed, TID_A_BITS, 0, m * (k // 32)).reshape(m, k // 32)
    a_scale = uniform_f16(seed, TID_A_SCALE, 0, m, 0.5, 1.5)
    w_bits = gen_binary_words(seed, n, k)
    scales = gen_scales(seed, n, k)
    return a_bits, a_scale, w_bits, scales


def sweep_tid(layer: int, j: int) -> int:
    return SWEEP_BASE + 16 * int(layer) + int(j)
