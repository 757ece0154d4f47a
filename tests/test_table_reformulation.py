"""The per-position table formulation of the one-token product, restated in
numpy and checked against the oracle (CPU only).

"Multiplication degenerates to addition and sign flip" (三值权重 page): the
one-token table kernels (csrc/gemv_lut.cu) do not expand codes; they
tabulate, for every byte position of a K slice, x . w over the byte's codes
for every byte value, and add one table entry per packed byte. This file
restates that formulation independently of the CUDA code (its own tables,
lane mapping and constants) and checks that it computes the oracle's y:

* ternary: slices of 640 codes (128 bytes, five whole groups); lane p owns
  bytes 4p..4p+3; the bytes that straddle a group edge (25, 51, 76, 102:
  codes 125..129, 255..259, 380..384, 510..514) keep their codes below the
  edge in the main table, and their codes above it are looked up by the
  byte's upper base-3 digits (index = byte / 3^k, a multiply-high) and
  handed, with the lane's later bytes, to the next lane;
* binary: slices of 1024 codes (eight whole groups), 256-entry tables, one
  group per lane.

It also pins the multiply-high constants ceil(2^16 / 3^k) * 2^16 as exact
for every byte value.
"""
import numpy as np
import pytest

import oracle
from sub_bit_weight_binary_b300 import synth

# (byte within the lane's word, digits below the group edge) per edge lane
EDGE = {6: (1, 3), 12: (3, 1), 19: (0, 4), 25: (2, 2)}


def f16(u16):
    return np.asarray(u16).view(np.float16).astype(np.float64)


def digits(e, n=5):
    return np.stack([(e // 3 ** i) % 3 for i in range(n)], axis=-1)


def test_multiply_high_index_is_exact():
    """byte / 3^k as the high word of byte * (ceil(2^16/3^k) << 16), for all
    256 byte values and k = 1..4 (the four edge bytes' digit splits)."""
    for k in range(1, 5):
        magic = (-(-65536 // 3 ** k)) << 16
        assert magic < 2 ** 32
        e = np.arange(256, dtype=np.uint64)
        assert np.array_equal((e * np.uint64(magic)) >> np.uint64(32), e // np.uint64(3 ** k))


def test_edge_bytes_are_the_group_straddlers():
    """In a 640-code slice exactly the bytes 25, 51, 76, 102 hold codes of two
    128-code groups, with 3, 1, 4 and 2 codes below the edge."""
    straddle = {}
    for b in range(128):
        lo = [c for c in range(5 * b, 5 * b + 5) if c // 128 == (5 * b) // 128]
        if len(lo) < 5:
            straddle[b] = len(lo)
    got = {4 * p + j: k for p, (j, k) in EDGE.items()}
    assert straddle == got == {25: 3, 51: 1, 76: 4, 102: 2}


def ternary_tables(xs):
    """Main tables T[byte][e] (codes below the position's group edge) and
    upper-digit tables H[lane][idx] of one 640-code slice, in float64."""
    d = digits(np.arange(243)) - 1                      # [243][5]
    xb = xs.reshape(128, 5)                             # codes of each byte
    mask = np.ones((128, 5))
    for p, (j, k) in EDGE.items():
        mask[4 * p + j, k:] = 0
    T = d @ (xb * mask).T                               # [243][128]
    H = np.zeros((32, 81))
    for p, (j, k) in EDGE.items():
        n = 3 ** (5 - k)
        dh = digits(np.arange(n), 5 - k) - 1           # [n][5-k]
        H[p, :n] = dh @ xb[4 * p + j, k:]
    return T, H


def ternary_by_tables(packed, scales, x, k):
    n = packed.shape[0]
    G = k // 128
    xf = f16(x.reshape(-1))
    sf = f16(scales)
    y = np.zeros(n)
    S = -(-k // 640)
    lane = np.arange(32)
    grp = (20 * lane) // 128                            # each lane's (lower) group
    js = np.array([EDGE.get(p, (0, 0))[0] for p in lane])
    kd = np.array([EDGE.get(p, (0, 0))[1] for p in lane])
    edge = np.array([p in EDGE for p in lane])
    for s in range(S):
        xs = np.zeros(640)
        seg = xf[640 * s: 640 * s + 640]
        xs[:len(seg)] = seg
        T, H = ternary_tables(xs)
        wb = np.zeros((n, 128), dtype=np.int64)         # bytes past the row read as zero
        part = packed[:, 128 * s: 128 * s + 128]
        wb[:, :part.shape[1]] = part
        sc = np.zeros((n, 5))
        for q in range(5):
            if 5 * s + q < G:
                sc[:, q] = sf[:, 5 * s + q]
        v = T[wb, np.arange(128)].reshape(n, 32, 4)     # [row][lane][byte of the word]
        above = edge[:, None] & (np.arange(4)[None, :] > js[:, None])   # wholly above the edge
        eb = wb.reshape(n, 32, 4)[:, lane, js]          # the edge byte of each lane
        idx = np.where(edge, eb // (3 ** kd), 0)
        h = H[lane[None, :], idx]
        hs = h + (v * above).sum(axis=2)                # handed to the next lane
        own = (v * ~above).sum(axis=2)
        hp = np.concatenate([np.zeros((n, 1)), hs[:, :-1]], axis=1)
        y += (sc[:, grp] * (own + hp)).sum(axis=1)
    return y


def binary_by_tables(packed, scales, x, k):
    n = packed.shape[0]
    G = k // 128
    xf = f16(x.reshape(-1))
    sf = f16(scales)
    e = np.arange(256)
    sign = ((e[:, None] >> np.arange(8)[None, :]) & 1) * 2.0 - 1.0   # [256][8]
    y = np.zeros(n)
    for s in range(-(-k // 1024)):
        xs = np.zeros(1024)
        seg = xf[1024 * s: 1024 * s + 1024]
        xs[:len(seg)] = seg
        T = sign @ xs.reshape(128, 8).T                 # [256][128]
        wb = np.zeros((n, 128), dtype=np.int64)
        part = packed[:, 128 * s: 128 * s + 128]
        wb[:, :part.shape[1]] = part
        sc = np.zeros((n, 8))
        for q in range(8):
            if 8 * s + q < G:
                sc[:, q] = sf[:, 8 * s + q]
        lanes = T[wb, np.arange(128)].reshape(n, 32, 4).sum(axis=2)
        y += (sc[:, np.arange(32) // 4] * lanes).sum(axis=1)
    return y


@pytest.mark.parametrize("n,k", [(48, 1280), (24, 1408), (16, 5120), (8, 17408)])
def test_ternary_tables_equal_the_oracle(n, k):
    """Whole slices, a partial last slice (K=1408: one group) and the decode
    shapes' K; float64 tables, so the only difference is rounding order."""
    codes = synth.gen_ternary_codes(700 + k % 97, n, k)
    packed = oracle.pack_ternary(codes)
    scales = synth.gen_scales(701, n, k)
    x = synth.gen_x(702, 1, k)
    y = ternary_by_tables(packed, scales, x, k)
    y_ref, nrm = oracle.linear(oracle.FMT_TERNARY, packed, scales, x)
    assert np.all(np.abs(y - y_ref[0]) <= 1e-9 * nrm[0] + 1e-300)


def test_ternary_tables_sparse_rows():
    """All-zero rows give exactly zero, single codes at the edge bytes are
    split correctly between their two groups."""
    n, k = 12, 1280
    codes = np.zeros((n, k), dtype=np.int8)
    for r, c in enumerate([125, 127, 128, 129, 255, 256, 383, 384, 511, 512, 640 + 128, 0]):
        codes[r, c] = 1 if r % 2 else -1
    codes[11] = 0
    packed = oracle.pack_ternary(codes)
    scales = synth.gen_scales(711, n, k)
    x = synth.gen_x(712, 1, k)
    y = ternary_by_tables(packed, scales, x, k)
    y_ref, nrm = oracle.linear(oracle.FMT_TERNARY, packed, scales, x)
    assert np.all(np.abs(y - y_ref[0]) <= 1e-12 * np.maximum(nrm[0], 1e-30))
    assert y[11] == 0.0


@pytest.mark.parametrize("n,k", [(32, 1024), (16, 3072), (8, 17408)])
def test_binary_tables_equal_the_oracle(n, k):
    words = synth.gen_binary_words(720 + k % 89, n, k)
    packed = words.view(np.uint8).reshape(n, -1)
    scales = synth.gen_scales(721, n, k)
    x = synth.gen_x(722, 1, k)
    y = binary_by_tables(packed, scales, x, k)
    y_ref, nrm = oracle.linear(oracle.FMT_BINARY, packed, scales, x)
    assert np.all(np.abs(y - y_ref[0]) <= 1e-9 * nrm[0] + 1e-300)
