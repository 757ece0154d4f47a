"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each pin_* function checks the oracle against something the oracle does not
compute the same way: the numbers the Bonsai pages print (tests/golden), a
closed form, an invariant, brute force through a second decoding route
(numpy unpackbits / integer division, then a dense float64 matmul), or
Python's own popcount. test_mutants_are_caught compiles deliberately broken
copies of oracle.c and checks that some pin rejects every one of them.
"""
import ctypes
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from sub_bit_weight_binary_b300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "pages_sizes.txt")

BIN, TER = oracle.FMT_BINARY, oracle.FMT_TERNARY


def golden():
    vals = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            vals[parts[0]] = float(parts[1])
    return vals


# ---- independent decoding routes (numpy), used only by the pins ----------

def np_decode_binary(packed_bytes, k):
    bits = np.unpackbits(np.ascontiguousarray(packed_bytes, dtype=np.uint8),
                         axis=1, bitorder="little")[:, :k]
    return bits.astype(np.int8) * 2 - 1


def np_decode_ternary(packed_bytes, k):
    b = np.ascontiguousarray(packed_bytes, dtype=np.int64)
    nbytes = (k + 4) // 5
    digits = np.stack([(b[:, :nbytes] // 3 ** i) % 3 for i in range(5)], axis=2)
    return (digits.reshape(b.shape[0], -1)[:, :k] - 1).astype(np.int8)


def f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dense(fmt, packed, scales, k):
    codes = np_decode_binary(packed, k) if fmt == BIN else np_decode_ternary(packed, k)
    s = np.repeat(f16(scales), 128, axis=1)
    return codes.astype(np.float64) * s


def rand_x(seed, m, k):
    return synth.gen_x(seed, m, k)


# ---- pins ----------------------------------------------------------------

def pin_half_to_double():
    h = np.arange(65536, dtype=np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(v)) for v in h[::7]])
    r = ref[::7]
    assert np.array_equal(np.isnan(got), np.isnan(r))
    ok = ~np.isnan(r)
    assert np.array_equal(got[ok], r[ok])
    for v in (0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x7C00, 0x8001, 0xFBFF):
        a, b = oracle.half_to_double(v), float(np.uint16(v).view(np.float16))
        assert a == b or (math.isnan(a) and math.isnan(b))


def pin_row_bytes():
    for k in (128, 256, 1024, 5120, 17408):
        assert oracle.row_bytes(BIN, k) == k // 8
    assert oracle.row_bytes(TER, 128) == 64      # 26 data bytes
    assert oracle.row_bytes(TER, 640) == 128     # exactly 128 data bytes
    assert oracle.row_bytes(TER, 5120) == 1024
    assert oracle.row_bytes(TER, 17408) == 3520  # 3482 data bytes
    for bad in (0, -128, 100, 129):
        assert oracle.row_bytes(BIN, bad) == -1
        assert oracle.row_bytes(TER, bad) == -1
    assert oracle.row_bytes(3, 128) == -1


def pin_page_sizes():
    g = golden()
    assert g["group_size"] == oracle.GROUP == 128
    for k in (128, 1024, 5120, 17408):
        bpw = (oracle.row_bytes(BIN, k) * 8 + 16 * k / 128) / k
        assert bpw == g["binary_bpw"]
    assert round(math.log2(3), 2) == g["ternary_info_bpw"]
    assert round(math.log2(3) + 16 / 128, 2) == g["ternary_bpw"]
    # the stored layout (5 codes per byte) is within 1% of the pages' figure
    k = 5120
    stored = (oracle.row_bytes(TER, k) * 8 + 16 * k / 128) / k
    assert abs(stored - g["ternary_bpw"]) / g["ternary_bpw"] < 0.01
    params = 27e9
    assert params * 2 / 1e9 == g["fp16_27b_gb"]
    ter_gb = params * g["ternary_bpw"] / 8 / 1e9
    assert ter_gb < g["ternary_27b_max_gb"]
    assert round(g["fp16_27b_gb"] / ter_gb) == g["ternary_27b_ratio"]
    assert round(params * g["binary_bpw"] / 8 / 1e9) == g["binary_27b_gb"]


def pin_binary_round_trip():
    for k, rows in ((128, 3), (640, 1), (5120, 3), (17408, 1), (128, 1024)):
        codes = synth.gen_binary_codes(11, rows, k)
        packed = oracle.pack_binary(codes)
        ref = np.packbits(((codes + 1) // 2).astype(np.uint8), axis=1, bitorder="little")
        assert np.array_equal(packed, ref)
        assert np.array_equal(oracle.unpack_binary(packed, k), codes)
        assert np.array_equal(np_decode_binary(packed, k), codes)


def pin_binary_single_hot():
    k = 256
    for pos in (0, 1, 7, 8, 31, 32, 100, 255):
        codes = -np.ones((1, k), dtype=np.int8)
        codes[0, pos] = 1
        words = oracle.pack_binary(codes).view("<u4")[0]
        expect = np.zeros(k // 32, dtype=np.uint32)
        expect[pos // 32] = np.uint32(1) << np.uint32(pos % 32)
        assert np.array_equal(words, expect), pos
    words = oracle.pack_binary(np.ones((1, k), dtype=np.int8)).view("<u4")[0]
    assert np.all(words == 0xFFFFFFFF)
    padded = oracle.pack_binary(np.ones((2, k), dtype=np.int8), k // 8 + 16)
    assert np.all(padded[:, k // 8:] == 0)


def pin_ternary_byte_values():
    k = 640
    for c, byte in ((-1, 0), (0, 121), (1, 242)):
        p = oracle.pack_ternary(np.full((1, k), c, dtype=np.int8))
        assert np.all(p == byte)
    for i in range(5):
        for b in (0, 7, 127):
            for sign in (1, -1):
                codes = np.zeros((1, k), dtype=np.int8)
                codes[0, 5 * b + i] = sign
                p = oracle.pack_ternary(codes)[0]
                assert p[b] == 121 + sign * 3 ** i
                assert np.all(np.delete(p, b) == 121)


def pin_ternary_all_bytes():
    k = 1280  # 256 data bytes
    vals = np.arange(256) % 243
    digits = np.stack([(vals // 3 ** i) % 3 for i in range(5)], axis=1)
    codes = (digits.reshape(1, -1) - 1).astype(np.int8)
    packed = oracle.pack_ternary(codes)
    assert np.array_equal(packed[0, :256], vals.astype(np.uint8))
    assert np.array_equal(oracle.unpack_ternary(packed, k), codes)
    for bad in (243, 250, 255):
        p = packed.copy()
        p[0, 3] = bad
        with pytest.raises(oracle.OracleError) as e:
            oracle.unpack_ternary(p, k)
        assert e.value.status == oracle.ERR_BAD_CODE


def pin_ternary_round_trip_and_padding():
    for k, rows in ((128, 3), (640, 2), (5120, 1), (17408, 1), (640, 1024)):
        codes = synth.gen_ternary_codes(5, rows, k)
        packed = oracle.pack_ternary(codes)
        assert packed.shape == (rows, oracle.row_bytes(TER, k))
        assert np.array_equal(oracle.unpack_ternary(packed, k), codes)
        assert np.array_equal(np_decode_ternary(packed, k), codes)
        nbytes = (k + 4) // 5
        assert np.all(packed[:, nbytes:] == 121)
        if k % 5:
            last = packed[:, nbytes - 1].astype(np.int64)
            for i in range(k - 5 * (nbytes - 1), 5):
                assert np.all((last // 3 ** i) % 3 == 1)  # padded codes are 0


def pin_bad_codes():
    c = np.ones((1, 128), dtype=np.int8)
    for bad in (0, 2, -2):
        c2 = c.copy()
        c2[0, 17] = bad
        with pytest.raises(oracle.OracleError) as e:
            oracle.pack_binary(c2)
        assert e.value.status == oracle.ERR_BAD_CODE
    for bad in (2, -2, 5):
        c2 = np.zeros((1, 128), dtype=np.int8)
        c2[0, 17] = bad
        with pytest.raises(oracle.OracleError) as e:
            oracle.pack_ternary(c2)
        assert e.value.status == oracle.ERR_BAD_CODE


def pin_all_plus_constant_scale():
    k, n = 1024, 3
    x = rand_x(1, 2, k)
    packed = np.full((n, k // 8), 0xFF, dtype=np.uint8)
    s = np.full((n, k // 128), np.float16(0.0371).view(np.uint16), dtype=np.uint16)
    y, nrm = oracle.linear(BIN, packed, s, x)
    expect = float(np.float16(0.0371)) * f16(x).sum(axis=1)
    assert np.allclose(y, expect[:, None], rtol=0, atol=1e-12 * nrm.max())
    assert np.allclose(nrm, float(np.float16(0.0371)) * np.abs(f16(x)).sum(axis=1)[:, None])


def pin_group_scales():
    k, n = 640, 2
    x = rand_x(2, 1, k)
    packed = np.full((n, k // 8), 0xFF, dtype=np.uint8)
    s = synth.gen_scales(3, n, k)
    y, nrm = oracle.linear(BIN, packed, s, x)
    xs = f16(x)[0].reshape(-1, 128).sum(axis=1)
    expect = (f16(s) * xs[None, :]).sum(axis=1)
    assert np.allclose(y[0], expect, rtol=0, atol=1e-12 * nrm.max())


def pin_zero_ternary():
    k, n = 640, 4
    x = rand_x(3, 2, k)
    packed = oracle.pack_ternary(np.zeros((n, k), dtype=np.int8))
    s = synth.gen_scales(4, n, k)
    y, nrm = oracle.linear(TER, packed, s, x)
    assert np.all(y == 0.0) and np.all(nrm == 0.0)


def pin_flip_and_scale():
    k, n = 512, 5
    x = rand_x(4, 3, k)
    w = synth.gen_binary_words(5, n, k)
    s = synth.gen_scales(6, n, k)
    y, _ = oracle.linear(BIN, w, s, x)
    y_flip, _ = oracle.linear(BIN, ~w, s, x)
    assert np.array_equal(y_flip, -y)
    for j in (1, 3):
        x2 = (f16(x) * 2.0 ** j).astype(np.float16).view(np.uint16)
        assert np.array_equal(f16(x2), f16(x) * 2.0 ** j)
        y2, _ = oracle.linear(BIN, w, s, x2)
        assert np.array_equal(y2, y * 2.0 ** j)


def pin_single_weight():
    k, n = 640, 3
    x = rand_x(5, 2, k)
    s = synth.gen_scales(7, n, k)
    for (n0, k0, sign) in ((1, 0, 1), (2, 129, -1), (0, 639, 1), (1, 384, -1)):
        codes = np.zeros((n, k), dtype=np.int8)
        codes[n0, k0] = sign
        y, _ = oracle.linear(TER, oracle.pack_ternary(codes), s, x)
        expect = np.zeros((2, n))
        expect[:, n0] = sign * f16(s)[n0, k0 // 128] * f16(x)[:, k0]
        assert np.array_equal(y, expect)


def pin_brute_force():
    for fmt in (BIN, TER):
        for (m, n, k) in ((1, 1, 128), (3, 4, 128), (2, 3, 256), (1, 2, 640)):
            x = rand_x(10 + m, m, k)
            s = synth.gen_scales(20 + n, n, k)
            if fmt == BIN:
                packed = synth.gen_binary_words(30 + k, n, k).view(np.uint8).reshape(n, -1)
            else:
                packed = oracle.pack_ternary(synth.gen_ternary_codes(40 + k, n, k))
            wd = dense(fmt, packed, s, k)
            ref = f16(x) @ wd.T
            nref = np.abs(f16(x)) @ np.abs(wd).T
            y, nrm = oracle.linear(fmt, packed, s, x)
            assert y.shape == (m, n)
            assert np.allclose(nrm, nref, rtol=1e-12, atol=0)
            assert np.all(np.abs(y - ref) <= 1e-12 * nref + 1e-300)
            # a sub-selection of rows and columns picks the same entries
            y2, _ = oracle.linear(fmt, packed, s, x, n_sel=[n - 1], m_sel=[m - 1])
            assert y2[0, 0] == y[m - 1, n - 1]


def pin_xnor():
    m, n, k = 3, 5, 512
    a_bits, a_s, w_bits, s = synth.gen_xnor_inputs(9, m, n, k)
    d, y, nrm = oracle.xnor(a_bits, a_s, w_bits, s, k)
    for i in range(m):
        for j in range(n):
            pc = [int(np.uint32(a_bits[i, t] ^ w_bits[j, t])).bit_count() for t in range(k // 32)]
            assert d[i, j] == k - 2 * sum(pc)
            dg = [128 - 2 * sum(pc[4 * g:4 * g + 4]) for g in range(k // 128)]
            ref = f16(a_s)[i] * sum(f16(s)[j, g] * dg[g] for g in range(k // 128))
            assert abs(y[i, j] - ref) <= 1e-12 * nrm[i, j]
            assert nrm[i, j] == abs(f16(a_s)[i]) * 128 * np.abs(f16(s)[j]).sum()
    # a = w gives D = K; a = NOT w gives D = -K
    d2, y2, _ = oracle.xnor(w_bits[:2], a_s[:2], w_bits, s, k)
    assert d2[0, 0] == k and d2[1, 1] == k
    assert abs(y2[0, 0] - f16(a_s)[0] * 128 * f16(s)[0].sum()) <= 1e-12
    d3, _, _ = oracle.xnor(~w_bits[:2], a_s[:2], w_bits, s, k)
    assert d3[0, 0] == -k and d3[1, 1] == -k


def pin_binarize():
    # closed form: the ramp x_k = (k - 63.5)/64 over one group is exact in
    # FP16; its first 64 entries are negative and sum |x| = 4096/64 = 64.
    k = 128
    ramp = ((np.arange(k) - 63.5) / 64).astype(np.float16)
    assert np.array_equal(ramp.astype(np.float64), (np.arange(k) - 63.5) / 64)
    bits, a_s = oracle.binarize(ramp.view(np.uint16)[None])
    assert bits.dtype == np.uint32 and bits.shape == (1, 4)
    assert list(bits[0]) == [0, 0, 0xFFFFFFFF, 0xFFFFFFFF]
    assert a_s[0] == 0.5
    # constant rows, and both zeros counting as +1 with a zero scale
    c = np.float16(0.3125)
    rows = np.stack([np.full(256, c), np.full(256, -c), np.zeros(256, np.float16),
                     np.full(256, np.float16(-0.0))]).astype(np.float16)
    assert np.signbit(rows[3]).all()
    bits, a_s = oracle.binarize(rows.view(np.uint16))
    assert np.all(bits[0] == 0xFFFFFFFF) and np.all(bits[1] == 0)
    assert np.all(bits[2] == 0xFFFFFFFF) and np.all(bits[3] == 0xFFFFFFFF)
    assert list(a_s) == [0.3125, 0.3125, 0.0, 0.0]
    # one negative entry clears exactly its own bit
    for pos in (0, 31, 32, 200):
        row = np.full((1, 256), np.float16(1.5))
        row[0, pos] = -2.0
        bits, a_s = oracle.binarize(row.astype(np.float16).view(np.uint16))
        expect = np.full(8, 0xFFFFFFFF, dtype=np.uint32)
        expect[pos // 32] ^= np.uint32(1) << np.uint32(pos % 32)
        assert np.array_equal(bits[0], expect) and a_s[0] == (255 * 1.5 + 2.0) / 256
    # a NaN compares false: code -1, and the scale is NaN
    row = np.ones((1, 128), np.float16)
    row[0, 5] = np.nan
    bits, a_s = oracle.binarize(row.view(np.uint16))
    assert bits[0, 0] == 0xFFFFFFFF ^ (1 << 5) and math.isnan(a_s[0])
    # invariants on random rows: the codes agree in sign with x, and the scale
    # is the least-squares one -- zero derivative of sum (x - alpha a)^2 and a
    # larger error on either side of it
    m, k = 5, 1024
    x = rand_x(21, m, k)
    bits, a_s = oracle.binarize(x)
    a = np_decode_binary(bits.view(np.uint8).reshape(m, -1), k).astype(np.float64)
    xv = f16(x)
    assert np.all(a * xv >= 0) and np.all(a[xv == 0] == 1)
    for i in range(m):
        err = lambda al: float(((xv[i] - al * a[i]) ** 2).sum())
        grad = float((a[i] * (xv[i] - a_s[i] * a[i])).sum())
        assert abs(grad) <= 1e-9 * np.abs(xv[i]).sum()
        assert err(a_s[i]) < err(a_s[i] * 1.001) and err(a_s[i]) < err(a_s[i] * 0.999)
    # composed with the XNOR product: weights equal to the codes give D = K
    s = synth.gen_scales(22, m, k)
    one = np.full(m, np.float16(1.0).view(np.uint16), dtype=np.uint16)
    d, y, _ = oracle.xnor(bits, one, bits, s, k)
    assert np.all(np.diag(d) == k)
    assert np.allclose(np.diag(y), 128 * f16(s).sum(axis=1), rtol=1e-12, atol=0)


def interleave_rows(gate, up):
    """[F][...] gate and up rows -> [2F][...], 16-row blocks of 8 gate rows
    followed by the 8 up rows of the same features (numpy reshapes only)."""
    f = gate.shape[0]
    g = gate.reshape(f // 8, 1, 8, *gate.shape[1:])
    u = up.reshape(f // 8, 1, 8, *up.shape[1:])
    return np.concatenate([g, u], axis=1).reshape(2 * f, *gate.shape[1:])


def pin_swiglu():
    # the stored-row mapping: g and u are the products of the separate matrices
    f, k, m = 24, 256, 3
    x = rand_x(31, m, k)
    for fmt in (BIN, TER):
        if fmt == BIN:
            gp = synth.gen_binary_words(32, f, k).view(np.uint8).reshape(f, -1)
            up = synth.gen_binary_words(33, f, k).view(np.uint8).reshape(f, -1)
        else:
            gp = oracle.pack_ternary(synth.gen_ternary_codes(32, f, k))
            up = oracle.pack_ternary(synth.gen_ternary_codes(33, f, k))
        gs, us = synth.gen_scales(34, f, k), synth.gen_scales(35, f, k)
        h, g, u, ng, nu = oracle.swiglu(fmt, interleave_rows(gp, up), interleave_rows(gs, us), x)
        g_ref, ng_ref = oracle.linear(fmt, gp, gs, x)
        u_ref, nu_ref = oracle.linear(fmt, up, us, x)
        assert np.array_equal(g, g_ref) and np.array_equal(u, u_ref)
        assert np.array_equal(ng, ng_ref) and np.array_equal(nu, nu_ref)
        # silu(g) - silu(-g) = g: flipping every gate weight changes h by g*u
        if fmt == BIN:
            h2, g2, _, _, _ = oracle.swiglu(fmt, interleave_rows(~gp, up), interleave_rows(gs, us), x)
            assert np.array_equal(g2, -g)
            assert np.allclose(h - h2, g * u, rtol=0, atol=1e-12 * np.abs(g * u).max())
        sel_h, _, _, _, _ = oracle.swiglu(fmt, interleave_rows(gp, up), interleave_rows(gs, us), x,
                                          f_sel=[f - 1, 0, 9], m_sel=[2, 0])
        assert np.array_equal(sel_h, h[np.ix_([2, 0], [f - 1, 0, 9])])
    # closed forms: x = 2^-7 everywhere and unit scales give g = +-1 over one
    # group of +-1 weights; sigma(1) = 1/(1 + 1/e) = 0.7310585786300049
    k, f = 128, 8
    x = np.full((1, k), np.float16(2.0 ** -7).view(np.uint16), dtype=np.uint16)
    ones = np.full((f, 1), np.float16(1.0).view(np.uint16), dtype=np.uint16)
    plus = np.full((f, k // 8), 0xFF, dtype=np.uint8)
    minus = np.zeros((f, k // 8), dtype=np.uint8)
    h, g, u, _, _ = oracle.swiglu(BIN, interleave_rows(plus, minus), interleave_rows(ones, ones), x)
    assert np.all(g == 1.0) and np.all(u == -1.0)
    assert np.allclose(h, -0.7310585786300049, rtol=1e-15, atol=0)
    h, g, u, _, _ = oracle.swiglu(BIN, interleave_rows(minus, plus), interleave_rows(ones, ones), x)
    assert np.allclose(h, -1.0 * (1.0 - 0.7310585786300049), rtol=1e-14, atol=0)
    # a large gate passes through (sigma = 1 in double), a zero gate gives 0
    big = np.full((f, 1), np.float16(64.0).view(np.uint16), dtype=np.uint16)
    h, g, u, _, _ = oracle.swiglu(BIN, interleave_rows(plus, plus), interleave_rows(big, ones), x)
    assert np.all(g == 64.0) and np.all(u == 1.0) and np.all(h == 64.0)
    zero = oracle.pack_ternary(np.zeros((f, k), dtype=np.int8))
    tplus = oracle.pack_ternary(np.ones((f, k), dtype=np.int8))
    h, g, u, ng, _ = oracle.swiglu(TER, interleave_rows(zero, tplus), interleave_rows(ones, ones), x)
    assert np.all(h == 0.0) and np.all(ng == 0.0) and np.all(u == 1.0)


def pin_hadamard():
    import scipy.linalg
    f = np.float16
    # worked example by hand: H4 [1,2,3,4] / 2 = [5, -1, -2, 0]
    x = np.array([[1, 2, 3, 4]], dtype=f).view(np.uint16)
    assert list(oracle.hadamard(x, 4)[0]) == [5.0, -1.0, -2.0, 0.0]
    assert np.allclose(oracle.hadamard(x, 2)[0], np.array([3, -1, 7, -1]) / np.sqrt(2),
                       rtol=1e-15, atol=0)
    # against scipy's Sylvester matrix (built by its own recursion), with signs
    for b, k in ((2, 64), (16, 64), (128, 384), (1024, 2048)):
        xr = rand_x(41 + b, 3, k)
        bits = synth.gen_binary_words(42 + b, 1, k)[0]
        sgn = np_decode_binary(bits.view(np.uint8)[None, :], k)[0].astype(np.float64)
        hm = scipy.linalg.hadamard(b).astype(np.float64) / np.sqrt(b)
        xs = (f16(xr) * sgn).reshape(3, k // b, b)
        ref = np.einsum("ij,rbj->rbi", hm, xs).reshape(3, k)
        got = oracle.hadamard(xr, b, bits)
        assert np.allclose(got, ref, rtol=0, atol=1e-12 * np.abs(f16(xr)).max() * np.sqrt(b))
        # orthonormal: the sum of squares of every block is kept
        assert np.allclose((got.reshape(3, -1, b) ** 2).sum(axis=2),
                           (f16(xr).reshape(3, -1, b) ** 2).sum(axis=2), rtol=1e-12, atol=0)
        # no sign vector means all +1
        assert np.array_equal(oracle.hadamard(xr, b), oracle.hadamard(xr, b, np.full(k // 32, 0xFFFFFFFF, np.uint32)))
    # unit vectors give the columns of H (entries +-b^-1/2), blocks do not mix
    b, k = 16, 48
    for j in (0, 5, 16 + 9, 47):
        e = np.zeros((1, k), dtype=f)
        e[0, j] = 1.0
        got = oracle.hadamard(e.view(np.uint16), b)[0]
        blk = j // b
        col = np.array([(-1) ** bin(i & (j % b)).count("1") for i in range(b)]) / 4.0
        assert np.array_equal(got[blk * b:(blk + 1) * b], col)
        assert np.all(np.delete(got, np.arange(blk * b, (blk + 1) * b)) == 0.0)
    # the rotation is its own inverse when b is an even power of two (exact
    # here: the first pass of these integer rows is again exact in FP16)
    xr = np.array([[3, -1, 4, 1, -5, 9, 2, -6, 5, 3, -5, 8, 9, -7, 9, 3]], dtype=f)
    once = oracle.hadamard(xr.view(np.uint16), 16)
    assert np.array_equal(once.astype(f).astype(np.float64), once)
    twice = oracle.hadamard(once.astype(f).view(np.uint16), 16)
    assert np.array_equal(twice, xr.astype(np.float64))
    # a cleared sign bit negates that input
    bits = np.full(1, 0xFFFFFFFF ^ (1 << 3), dtype=np.uint32)
    xr32 = rand_x(43, 1, 32)
    neg = xr32.copy()
    neg[0, 3] ^= 0x8000
    assert np.array_equal(oracle.hadamard(xr32, 32, bits), oracle.hadamard(neg, 32))


def pin_compare_rule():
    ref = np.array([1.0, 1.0, 0.0, 1.0, 1.0])
    nrm = np.array([10.0, 10.0, 0.0, 10.0, 10.0])
    good = np.array([1.0, 1.015, -0.0, 0.99, 1.0], dtype=np.float16).view(np.uint16)
    bad, first, worst = oracle.compare_f16(good, ref, nrm)
    assert bad == 0 and first == -1 and worst <= 2e-3
    y = good.copy()
    y[1] = np.float16(1.03).view(np.uint16)      # 3e-3 of norm
    y[2] = np.float16(1e-7).view(np.uint16)      # zero-norm entry must be 0
    y[4] = np.float16(np.nan).view(np.uint16)
    bad, first, _ = oracle.compare_f16(y, ref, nrm)
    assert bad == 3 and first == 1


PINS = [pin_half_to_double, pin_row_bytes, pin_page_sizes, pin_binary_round_trip,
        pin_binary_single_hot, pin_ternary_byte_values, pin_ternary_all_bytes,
        pin_ternary_round_trip_and_padding, pin_bad_codes,
        pin_all_plus_constant_scale, pin_group_scales, pin_zero_ternary,
        pin_flip_and_scale, pin_single_weight, pin_brute_force, pin_xnor,
        pin_binarize, pin_swiglu, pin_hadamard, pin_compare_rule]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_lib):
    pin()


# Each mutant is a plausible slip in oracle.c; some pin must reject it.
MUTANTS = {
    "bit_polarity": ("if (c == 1)\n          word", "if (c == -1)\n          word"),
    "bit_order": ("word |= (uint32_t)1 << i;", "word |= (uint32_t)1 << (31 - i);"),
    "unpack_polarity": ("((word >> i) & 1u) ? 1 : -1", "((word >> i) & 1u) ? -1 : 1"),
    "trit_digit_order": ("int64_t kk = 5 * b + i;\n        int c = 0;",
                         "int64_t kk = 5 * b + (4 - i);\n        int c = 0;"),
    "trit_offset": ("value = 3 * value + (c + 1);", "value = 3 * value + (1 - c);"),
    "unpack_trit_order": ("if (kk < k) codes[r * k + kk] = (int8_t)(digit - 1);",
                          "if (kk < k) codes[r * k + (5 * b + 4 - i)] = (int8_t)(digit - 1);"),
    "group_index": ("scales[nn * groups + kk / GROUP]", "scales[nn * groups + kk / 64 % groups]"),
    "scale_divides": ("double t = xv * sv * (double)w[kk];", "double t = xv / sv * (double)w[kk];"),
    "dropped_abs": ("nrm += fabs(t);", "nrm += t;"),
    "transposed_x": ("double xv = oracle_half_to_double(x[mm * k + kk]);",
                     "double xv = oracle_half_to_double(x[kk * m % (m * k) + mm]);"),
    "half_bias": ("ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)"),
    "half_subnormal": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "xnor_group_scale": ("acc += sg * (double)dg;", "acc += sg * (double)total;"),
    "xnor_sign": ("dg += (int64_t)a[kk] * (int64_t)w[kk];", "dg -= (int64_t)a[kk] * (int64_t)w[kk];"),
    "ter_pad_bytes": ("return 64 * ((data + 63) / 64);", "return 16 * ((data + 15) / 16);"),
    "binarize_zero_sign": ("a[kk] = (v >= 0.0) ? 1 : -1;", "a[kk] = (v > 0.0) ? 1 : -1;"),
    "binarize_no_abs": ("sum += fabs(v);", "sum += v;"),
    "binarize_squares": ("sum += fabs(v);", "sum += v * v;"),
    "binarize_divisor": ("a_scale[r] = sum / (double)k;", "a_scale[r] = sum / (double)(k - 1);"),
    "swiglu_sign": ("h[o] = gv / (1.0 + exp(-gv)) * uv;", "h[o] = gv / (1.0 + exp(gv)) * uv;"),
    "swiglu_swapped": ("h[o] = gv / (1.0 + exp(-gv)) * uv;", "h[o] = uv / (1.0 + exp(-uv)) * gv;"),
    "swiglu_block": ("rows[j] = 16 * (f / 8) + f % 8;", "rows[j] = 8 * (f / 8) + f % 8;"),
    "swiglu_up_offset": ("rows[f_cnt + j] = rows[j] + 8;", "rows[f_cnt + j] = rows[j] + 1;"),
    "hadamard_or": ("(unsigned long long)(i & j)", "(unsigned long long)(i | j)"),
    "hadamard_norm": ("const double scale = 1.0 / sqrt((double)block);",
                      "const double scale = 1.0 / (double)block;"),
    "hadamard_sign_index": ("(sign_bits[kk >> 3] >> (kk & 7)) & 1", "(sign_bits[kk >> 3] >> (j & 7)) & 1"),
    "hadamard_block_base": ("const int64_t kk = b0 + j;", "const int64_t kk = j;"),
    "ter_bad_byte": ("if (value > 242) return O_ERR_BAD_CODE;", "if (value > 255) return O_ERR_BAD_CODE;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, tmp_path, oracle_lib):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = open(oracle.SRC, encoding="utf-8").read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "mutation anchor not found exactly once: " + name
    path = tmp_path / ("oracle_%s.c" % name)
    path.write_text(src.replace(old, new), encoding="utf-8")
    so = tmp_path / ("liboracle_%s.so" % name)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so),
                           str(path), "-lm"])
    mutant = oracle.configure(ctypes.CDLL(str(so)))
    prev = oracle.use_library(mutant)
    caught = []
    try:
        for pin in PINS:
            try:
                pin()
            except (AssertionError, oracle.OracleError, ValueError, pytest.fail.Exception):
                caught.append(pin.__name__)
    finally:
        oracle.use_library(prev)
    assert caught, "no pin caught mutant " + name
