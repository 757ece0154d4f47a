"""CUDA path against the CPU oracle on the same seeded inputs (needs a GPU).

Byte-exact for packing, bit-exact for the XNOR integer dot, and
|y - y_ref| <= 2e-3 * sum|x*s*w| for every FP16 output. Shapes span several
tiles plus ragged tails; full-size workloads are checked on sampled outputs
(tile edges included) that the oracle computes one by one."""
import numpy as np
import pytest

import oracle
import sub_bit_weight_binary_b300 as sb
from sub_bit_weight_binary_b300 import synth
from gpu_util import Guarded, assert_close, assert_swiglu_close, dev, host, torch, weights

pytestmark = pytest.mark.gpu
BIN, TER = sb.BONSAI_FMT_BINARY, sb.BONSAI_FMT_TERNARY


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    t = torch()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from sub_bit_weight_binary_b300 import build
    build.build()
    sb.lib()
    oracle.lib()
    yield
    assert sb.bonsai_check_async() == 0


# ---------------------------------------------------------------- generator
def test_device_generator_matches_host():
    from sub_bit_weight_binary_b300 import synth_device as sd
    t = torch()
    n = 300001
    out = t.empty(n, dtype=t.int32, device="cuda")
    sd.bits32(11, 5, 1000, out)
    assert np.array_equal(host(out).view(np.uint32), synth.bits32(11, 5, 1000, n))
    c = t.empty(n, dtype=t.int8, device="cuda")
    sd.ternary_codes(12, 6, 77, c)
    assert np.array_equal(host(c), synth.ternary_codes(12, 6, 77, n))
    sd.binary_codes(13, 7, 0, c)
    assert np.array_equal(host(c), synth.binary_codes(13, 7, 0, n))
    h = t.empty(n, dtype=t.float16, device="cuda")
    sd.uniform_f16(14, 8, 5, 0.01, 0.05, h)
    assert np.array_equal(host(h), synth.uniform_f16(14, 8, 5, n, 0.01, 0.05))


# --------------------------------------------------------------------- pack
PACK_SHAPES = [(1, 128, 0), (3, 640, 0), (17, 5120, 0), (5, 17408, 0), (1024, 1024, 0),
               (7, 256, 64)]


@pytest.mark.parametrize("rows,k,pad", PACK_SHAPES)
def test_pack_binary_bytes(rows, k, pad):
    t = torch()
    codes = synth.gen_binary_codes(21, rows, k)
    rb = k // 8 + pad
    out = Guarded((rows, rb), t.uint8)
    sb.bonsai_pack_binary(dev(codes), out.t)
    assert sb.bonsai_check_async() == 0
    assert np.array_equal(host(out.t), oracle.pack_binary(codes, rb))
    out.check()


@pytest.mark.parametrize("rows,k,pad", PACK_SHAPES)
def test_pack_ternary_bytes(rows, k, pad):
    t = torch()
    codes = synth.gen_ternary_codes(22, rows, k)
    rb = sb.bonsai_packed_row_bytes(TER, k) + pad
    out = Guarded((rows, rb), t.uint8)
    sb.bonsai_pack_ternary(dev(codes), out.t)
    assert sb.bonsai_check_async() == 0
    assert np.array_equal(host(out.t), oracle.pack_ternary(codes, rb))
    out.check()


def test_pack_reports_bad_codes():
    t = torch()
    codes = synth.gen_binary_codes(23, 4, 256)
    codes[2, 77] = 0
    out = t.empty((4, 32), dtype=t.uint8, device="cuda")
    sb.bonsai_pack_binary(dev(codes), out)
    assert sb.STATUS[sb.bonsai_check_async()] == "BONSAI_ERR_BAD_CODE"
    assert sb.bonsai_check_async() == 0  # the status word was cleared
    tc = synth.gen_ternary_codes(24, 4, 256)
    tc[1, 3] = 2
    out2 = t.empty((4, 64), dtype=t.uint8, device="cuda")
    sb.bonsai_pack_ternary(dev(tc), out2)
    assert sb.STATUS[sb.bonsai_check_async()] == "BONSAI_ERR_BAD_CODE"
    assert sb.bonsai_check_async() == 0


# --------------------------------------------------------------------- GEMV
GEMV_CASES = [
    (BIN, 1024, 1024),    # binary decode workload (M=1, K=N=1024)
    (BIN, 1, 128), (BIN, 17, 640), (BIN, 33, 5120), (BIN, 1000, 1024),
    (BIN, 16, 17408), (BIN, 5120, 5120), (BIN, 301, 9216),
    (BIN, 7, 384), (BIN, 50, 8192), (BIN, 2000, 8320),  # subset-sum kernel: odd G, largest K; past it
    (TER, 17408, 5120),   # ternary decode workload (M=1, K=5120, N=17408)
    (TER, 1, 128), (TER, 17, 640), (TER, 33, 5120), (TER, 40, 17408),
    (TER, 5120, 17408), (TER, 300, 1280), (TER, 129, 384),
    # the decode sweep's stacked q/k/v and gate/up matrices
    (BIN, 15360, 5120), (TER, 15360, 5120), (BIN, 34816, 5120), (TER, 34816, 5120),
    # rows too long for the decode kernel's x table: the tensor-core fallback
    (TER, 20, 65536), (BIN, 20, 131072), (TER, 3, 1 << 20),
]


@pytest.mark.parametrize("fmt,n,k", GEMV_CASES)
def test_gemv(fmt, n, k):
    t = torch()
    w, packed, scales = weights(fmt, 100 + n % 97, n, k)
    x = synth.gen_x(31 + k % 13, 1, k)
    y = Guarded((n,), t.float16)
    sb.bonsai_gemv(w, dev(x[0]), y.t)
    assert sb.bonsai_check_async() == 0
    y_ref, nrm = oracle.linear(fmt, packed, scales, x)
    assert_close(host(y.t), y_ref[0], nrm[0], "gemv fmt=%d n=%d k=%d" % (fmt, n, k))
    y.check()


@pytest.mark.parametrize("fmt", [BIN, TER])
def test_gemv_wide_range_activations(fmt):
    """x spanning many binades (1e-4 .. 1e3, both signs) and exact zeros:
    the one-token kernels (subset-sum tables in FP32 for binary) stay within
    the bound of every output."""
    t = torch()
    n, k = 333, 5120
    w, packed, scales = weights(fmt, 12, n, k)
    rng = np.random.default_rng(5)
    mag = 10.0 ** rng.uniform(-4, 3, size=k)
    xv = (mag * rng.choice([-1.0, 1.0], size=k)).astype(np.float16)
    xv[rng.integers(0, k, size=k // 10)] = 0
    x = xv.view(np.uint16)[None, :]
    y = Guarded((n,), t.float16)
    sb.bonsai_gemv(w, dev(x[0]), y.t)
    assert sb.bonsai_check_async() == 0
    y_ref, nrm = oracle.linear(fmt, packed, scales, x)
    assert_close(host(y.t), y_ref[0], nrm[0], "wide-range x fmt=%d" % fmt)
    y.check()


@pytest.mark.parametrize("fmt", [BIN, TER])
def test_gemv_prefetch_flag_same_result(fmt):
    t = torch()
    n, k = 777, 5120
    w, packed, scales = weights(fmt, 7, n, k)
    x = dev(synth.gen_x(8, 1, k)[0])
    y0 = t.empty(n, dtype=t.float16, device="cuda")
    y1 = t.empty(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv(w, x, y0)
    w.flags = sb.BONSAI_WEIGHTS_PREFETCH
    sb.bonsai_gemv(w, x, y1)
    assert sb.bonsai_check_async() == 0
    assert t.equal(y0.view(t.int16), y1.view(t.int16))


def test_gemv_special_values():
    """All +1 binary rows with a constant scale give s*sum(x); flipping every
    bit negates; all-zero ternary rows give exactly 0."""
    t = torch()
    n, k = 48, 1024
    x = synth.gen_x(9, 1, k)
    s = np.full((n, k // 128), np.float16(0.03125).view(np.uint16), dtype=np.uint16)
    ones = np.full((n, k // 8), 0xFF, dtype=np.uint8)
    w = sb.Weights(BIN, n, k, dev(ones), dev(s))
    y = t.empty(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv(w, dev(x[0]), y)
    w2 = sb.Weights(BIN, n, k, dev(~ones), dev(s))
    y2 = t.empty(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv(w2, dev(x[0]), y2)
    assert sb.bonsai_check_async() == 0
    ref = 0.03125 * x.view(np.float16).astype(np.float64).sum()
    got = host(y).view(np.float16).astype(np.float64)
    nrm = 0.03125 * np.abs(x.view(np.float16).astype(np.float64)).sum()
    assert np.all(np.abs(got - ref) <= 2e-3 * nrm)
    assert np.array_equal(host(y2).view(np.float16).astype(np.float64), -got)
    zc = np.zeros((n, k), dtype=np.int8)
    packed = t.empty((n, sb.bonsai_packed_row_bytes(TER, k)), dtype=t.uint8, device="cuda")
    sb.bonsai_pack_ternary(dev(zc), packed)
    wz = sb.Weights(TER, n, k, packed, dev(s))
    yz = t.empty(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv(wz, dev(x[0]), yz)
    assert sb.bonsai_check_async() == 0
    assert np.all(host(yz).view(np.float16) == 0)


@pytest.mark.parametrize("fmt", [BIN, TER])
@pytest.mark.parametrize("m", [1, 3, 300])
def test_degenerate_scales_and_inputs(fmt, m):
    """Zero scales or zero activations give exactly +-0 (the norm is 0);
    negating every scale negates every output bit-exactly (s*w is exact and
    negation commutes with round-to-nearest), on the decode (m <= 8) and the
    tensor-core (m = 300) paths."""
    t = torch()
    n, k = 200, 1280
    w, packed, scales = weights(fmt, 230 + m, n, k)
    x = synth.gen_x(231 + m, m, k)

    def run(sc, xv):
        ww = sb.Weights(fmt, n, k, w.packed, dev(sc))
        y = t.empty((m, n), dtype=t.float16, device="cuda")
        sb.bonsai_gemm(ww, dev(xv), y)
        assert sb.bonsai_check_async() == 0
        return host(y)

    zero_s = np.zeros_like(scales)
    assert np.all((run(zero_s, x) & 0x7FFF) == 0)
    assert np.all((run(scales, np.zeros_like(x)) & 0x7FFF) == 0)
    y = run(scales, x)
    y_neg = run(scales ^ np.uint16(0x8000), x)
    assert np.array_equal(y_neg & 0x7FFF, y & 0x7FFF)       # same magnitudes
    nz = (y & 0x7FFF) != 0                                    # an exact 0 may keep its sign
    assert np.array_equal(y_neg[nz], y[nz] ^ np.uint16(0x8000))
    # one group's scales zeroed: that group contributes nothing
    part = scales.copy()
    part[:, 3] = 0
    y_ref, nrm = oracle.linear(fmt, packed, part, x)
    assert_close(run(part, x), y_ref, nrm, "one zero group")


def _sparse_ternary_codes(seed, n, k, per_mille):
    """Seeded ternary codes with `per_mille`/1000 of them nonzero (+-1 equally
    likely), from the counter-based generator's raw words."""
    w = synth.words(seed, 0x51, 0, n * k)
    keep = (w >> np.uint64(54)) < np.uint64(per_mille * 1024 // 1000)
    sign = np.where((w & np.uint64(1)) == 1, 1, -1)
    return np.where(keep, sign, 0).astype(np.int8).reshape(n, k)


def _ternary_from_codes(codes, seed):
    t = torch()
    n, k = codes.shape
    rb = sb.bonsai_packed_row_bytes(TER, k)
    packed_gpu = t.empty((n, rb), dtype=t.uint8, device="cuda")
    sb.bonsai_pack_ternary(dev(codes), packed_gpu)
    scales = synth.gen_scales(seed, n, k)
    return sb.Weights(TER, n, k, packed_gpu, dev(scales)), oracle.pack_ternary(codes), scales


@pytest.mark.parametrize("per_mille", [100, 20, 5])
@pytest.mark.parametrize("m", [1, 3])
def test_sparse_ternary(per_mille, m):
    """Rows with few nonzero weights: every output must still meet the bound
    against its own (small) norm, so zero codes may add nothing to the error."""
    n, k = 300, 5120
    codes = _sparse_ternary_codes(60 + per_mille, n, k, per_mille)
    w, packed, scales = _ternary_from_codes(codes, 61)
    x = synth.gen_x(62, m, k)
    y = Guarded((m, n), torch().float16)
    sb.bonsai_gemm(w, dev(x), y.t)
    assert sb.bonsai_check_async() == 0
    y_ref, nrm = oracle.linear(TER, packed, scales, x)
    assert_close(host(y.t), y_ref, nrm, "sparse ternary %d/1000 m=%d" % (per_mille, m))
    y.check()


def test_one_nonzero_ternary_per_row():
    """Each row holds a single nonzero code (at a seeded position and sign);
    y must be s*x[k] to the bound, with all other codes contributing nothing."""
    n, k = 512, 5120
    r = synth.words(70, 0x52, 0, n)
    pos = (r % np.uint64(k)).astype(np.int64)
    codes = np.zeros((n, k), dtype=np.int8)
    codes[np.arange(n), pos] = np.where((r >> np.uint64(63)) == 1, 1, -1)
    w, packed, scales = _ternary_from_codes(codes, 71)
    x = synth.gen_x(72, 1, k)
    y = torch().empty(n, dtype=torch().float16, device="cuda")
    sb.bonsai_gemv(w, dev(x[0]), y)
    assert sb.bonsai_check_async() == 0
    y_ref, nrm = oracle.linear(TER, packed, scales, x)
    assert_close(host(y), y_ref[0], nrm[0], "one nonzero per row")


# ------------------------------------------------------------ GEMM, small m
@pytest.mark.parametrize("fmt", [BIN, TER])
@pytest.mark.parametrize("m,n,k", [(2, 300, 1024), (5, 1024, 5120), (8, 129, 640), (3, 64, 17408),
                                   # ternary 5..8 tokens in one launch (one B column per
                                   # token), and a K whose x tables force two launches
                                   (6, 400, 5120), (7, 33, 1280), (5, 50, 17408)])
def test_gemm_few_tokens(fmt, m, n, k):
    t = torch()
    w, packed, scales = weights(fmt, 40 + m, n, k)
    x = synth.gen_x(50 + m, m, k)
    y = Guarded((m, n), t.float16)
    sb.bonsai_gemm(w, dev(x), y.t)
    assert sb.bonsai_check_async() == 0
    y_ref, nrm = oracle.linear(fmt, packed, scales, x)
    assert_close(host(y.t), y_ref, nrm, "gemm m=%d" % m)
    y.check()


# ------------------------------------------------------- GEMM, tensor cores
@pytest.mark.parametrize("fmt", [BIN, TER])
@pytest.mark.parametrize("m,n,k", [(9, 128, 128), (300, 200, 640), (512, 384, 1024),
                                   (257, 130, 5120), (256, 256, 320 * 4), (130, 96, 17408),
                                   (600, 136, 640), (1000, 130, 256), (1536, 272, 384)])
def test_gemm_tensor_core(fmt, m, n, k):
    t = torch()
    w, packed, scales = weights(fmt, 60 + m, n, k)
    x = synth.gen_x(70 + m, m, k)
    y = Guarded((m, n), t.float16)
    sb.bonsai_gemm(w, dev(x), y.t)
    assert sb.bonsai_check_async() == 0
    y_ref, nrm = oracle.linear(fmt, packed, scales, x)
    assert_close(host(y.t), y_ref, nrm, "gemm m=%d n=%d k=%d" % (m, n, k))
    y.check()


@pytest.mark.parametrize("m", [300, 600, 1000])
def test_gemm_wide_tiles(m):
    """Ternary products with enough feature tiles to take 512-token tiles
    (n = 17040: 134 tiles, the last one ragged), token counts that leave the
    second 256-token half partly or wholly empty; sampled outputs."""
    t = torch()
    n, k = 17040, 256
    w, packed, scales = weights(TER, 210 + m, n, k)
    x = synth.gen_x(211 + m, m, k)
    y = Guarded((m, n), t.float16)
    sb.bonsai_gemm(w, dev(x), y.t)
    assert sb.bonsai_check_async() == 0
    ms = sample_idx(m, [0, 255, 256, 299, 511, 512, 767, 768, m - 1], 20, 12)
    ns = sample_idx(n, [0, 127, 128, n - 17, n - 16, n - 1], 60, 13)
    y_ref, nrm = oracle.linear(TER, packed, scales, x, n_sel=ns, m_sel=ms)
    assert_close(host(y.t)[np.ix_(ms, ns)], y_ref, nrm, "wide tiles m=%d" % m)
    y.check()


@pytest.mark.parametrize("n,m", [(17040, 9), (17040, 300), (17040, 600), (16900, 257)])
def test_gemm_tall_tiles(n, m):
    """Binary products with enough feature tiles to take 256-feature tiles:
    the last tile's second 128-row half partly (n = 17040) or wholly
    (n = 16900) past n; ragged token tiles; sampled outputs."""
    t = torch()
    k = 384
    w, packed, scales = weights(BIN, 220 + m, n, k)
    x = synth.gen_x(221 + m, m, k)
    y = Guarded((m, n), t.float16)
    sb.bonsai_gemm(w, dev(x), y.t)
    assert sb.bonsai_check_async() == 0
    ms = sample_idx(m, [0, 8, 255, 256, m - 1], 16, 14)
    ns = sample_idx(n, [0, 127, 128, 255, 256, 16895, 16896, 16900 - 1, n - 17, n - 16, n - 1], 60, 15)
    y_ref, nrm = oracle.linear(BIN, packed, scales, x, n_sel=ns, m_sel=ms)
    assert_close(host(y.t)[np.ix_(ms, ns)], y_ref, nrm, "tall tiles n=%d m=%d" % (n, m))
    y.check()


def sample_idx(total, edges, count, seed):
    rng = np.random.default_rng(seed)
    idx = set(int(e) for e in edges if 0 <= e < total)
    idx.update(int(v) for v in rng.integers(0, total, count))
    return np.array(sorted(idx), dtype=np.int64)


@pytest.mark.parametrize("fmt", [BIN, TER])
@pytest.mark.parametrize("m", [512, 4096])
def test_gemm_prefill_workload_sampled(fmt, m):
    """The prefill / DiT workload (K=5120, N=17408) at full size, checked on
    sampled outputs including every tile edge row and column."""
    t = torch()
    n, k = 17408, 5120
    w, packed, scales = weights(fmt, 80, n, k)
    x = synth.gen_x(81, m, k)
    y = Guarded((m, n), t.float16)
    sb.bonsai_gemm(w, dev(x), y.t)
    assert sb.bonsai_check_async() == 0
    ms = sample_idx(m, [0, 1, 127, 128, 255, 256, m - 1], 40, 1)
    ns = sample_idx(n, [0, 1, 127, 128, 255, 256, n - 129, n - 128, n - 1], 60, 2)
    y_ref, nrm = oracle.linear(fmt, packed, scales, x, n_sel=ns, m_sel=ms)
    yg = host(y.t)[np.ix_(ms, ns)]
    assert_close(yg, y_ref, nrm, "gemm workload m=%d" % m)
    y.check()


# --------------------------------------------------------------------- XNOR
# popc=False: the tensor-core kernel; True: the literal XOR + popcount kernel
@pytest.mark.parametrize("popc", [False, True])
@pytest.mark.parametrize("m,n,k", [(64, 256, 4096), (70, 100, 640), (1, 1, 128), (130, 65, 1024),
                                   (300, 260, 2048), (129, 129, 128)])
def test_xnor_full(m, n, k, popc):
    t = torch()
    a_bits, a_s, w_bits, s = synth.gen_xnor_inputs(90 + m, m, n, k)
    w = sb.Weights(BIN, n, k, dev(w_bits.view(np.uint8).reshape(n, -1)), dev(s))
    d = Guarded((m, n), t.int32)
    y = Guarded((m, n), t.float16)
    sb.bonsai_xnor_gemm(dev(a_bits.view(np.int32)), dev(a_s), w, d.t, y.t, popc=popc)
    assert sb.bonsai_check_async() == 0
    d_ref, y_ref, nrm = oracle.xnor(a_bits, a_s, w_bits, s, k)
    assert np.array_equal(host(d.t).astype(np.int64), d_ref)
    assert_close(host(y.t), y_ref, nrm, "xnor")
    d.check()
    y.check()


@pytest.mark.parametrize("popc", [False, True])
def test_xnor_workload(popc):
    """XNOR workload M=512, K=4096, N=4096: D sampled against the oracle and
    every D checked against the popcount route of numpy; Y sampled. Both
    kernels (tensor cores, XOR + popcount)."""
    t = torch()
    m, n, k = 512, 4096, 4096
    a_bits, a_s, w_bits, s = synth.gen_xnor_inputs(95, m, n, k)
    w = sb.Weights(BIN, n, k, dev(w_bits.view(np.uint8).reshape(n, -1)), dev(s))
    d = Guarded((m, n), t.int32)
    y = Guarded((m, n), t.float16)
    sb.bonsai_xnor_gemm(dev(a_bits.view(np.int32)), dev(a_s), w, d.t, y.t, popc=popc)
    d_only = t.empty((m, n), dtype=t.int32, device="cuda")
    sb.bonsai_xnor_gemm(dev(a_bits.view(np.int32)), dev(a_s), w, d_only, None, popc=popc)
    y_only = t.empty((m, n), dtype=t.float16, device="cuda")
    sb.bonsai_xnor_gemm(dev(a_bits.view(np.int32)), dev(a_s), w, None, y_only, popc=popc)
    assert sb.bonsai_check_async() == 0
    if not popc:  # the two kernels agree: D bit for bit, Y within the sum of both bounds
        d_p = t.empty((m, n), dtype=t.int32, device="cuda")
        y_p = t.empty((m, n), dtype=t.float16, device="cuda")
        sb.bonsai_xnor_gemm(dev(a_bits.view(np.int32)), dev(a_s), w, d_p, y_p, popc=True)
        assert sb.bonsai_check_async() == 0
        assert t.equal(d.t, d_p)
    dg = host(d.t)
    assert np.array_equal(dg, host(d_only))
    assert np.array_equal(host(y.t), host(y_only))
    ms = sample_idx(m, [0, 63, 64, m - 1], 30, 3)
    ns = sample_idx(n, [0, 63, 64, n - 1], 40, 4)
    d_ref, y_ref, nrm = oracle.xnor(a_bits, a_s, w_bits, s, k, n_sel=ns, m_sel=ms)
    assert np.array_equal(dg[np.ix_(ms, ns)].astype(np.int64), d_ref)
    assert_close(host(y.t)[np.ix_(ms, ns)], y_ref, nrm, "xnor workload")
    for i in range(0, m, 64):  # all of D, 64 rows at a time
        x = np.bitwise_xor(a_bits[i:i + 64, None, :], w_bits[None, :, :])
        ref = k - 2 * np.bitwise_count(x).sum(axis=2, dtype=np.int64)
        assert np.array_equal(dg[i:i + 64].astype(np.int64), ref)
    d.check()
    y.check()


@pytest.mark.parametrize("fmt", [BIN, TER])
def test_gemm_down_projection_sampled(fmt):
    """The down projection of a prefill layer (M=512, K=17408, N=5120) at
    full size, sampled outputs."""
    t = torch()
    m, n, k = 512, 5120, 17408
    w, packed, scales = weights(fmt, 180 + fmt, n, k)
    x = synth.gen_x(181, m, k)
    y = Guarded((m, n), t.float16)
    sb.bonsai_gemm(w, dev(x), y.t)
    assert sb.bonsai_check_async() == 0
    ms = sample_idx(m, [0, 255, 256, m - 1], 10, 9)
    ns = sample_idx(n, [0, 127, 128, n - 1], 40, 10)
    y_ref, nrm = oracle.linear(fmt, packed, scales, x, n_sel=ns, m_sel=ms)
    assert_close(host(y.t)[np.ix_(ms, ns)], y_ref, nrm, "down projection")
    y.check()


@pytest.mark.parametrize("fmt,n,k", [(TER, 17408, 5120), (BIN, 1024, 1024), (TER, 33, 640),
                                     (TER, 20, 65536)])  # last: tensor-core fallback, y into host memory
def test_gemv_host_buffers(fmt, n, k):
    """bonsai_gemv_host (host x in, host y out, one call) gives the bits of
    bonsai_gemv and meets the oracle's bound; pinned and pageable host memory."""
    t = torch()
    w, packed, scales = weights(fmt, 200 + n, n, k)
    x = synth.gen_x(201, 1, k)[0]
    y_ref_dev = t.empty(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv(w, dev(x), y_ref_dev)
    for pinned in (True, False):
        x_host = t.from_numpy(x.view(np.float16).copy())
        y_host = t.zeros(n, dtype=t.float16)
        if pinned:
            x_host, y_host = x_host.pin_memory(), y_host.pin_memory()
        x_dev = t.empty(k, dtype=t.float16, device="cuda")
        y_dev = t.empty(n, dtype=t.float16, device="cuda")
        sb.bonsai_gemv_host(w, x_host, x_dev, y_dev, y_host)
        assert sb.bonsai_check_async() == 0
        yh = y_host.numpy().view(np.uint16)
        assert np.array_equal(yh, host(y_ref_dev))
        ns = sample_idx(n, [0, n - 1], 64, 11)
        y_ref, nrm = oracle.linear(fmt, packed, scales, x, n_sel=ns)
        assert_close(yh[ns][None, :], y_ref, nrm, "gemv host buffers")
        if pinned:  # the prepared (graph-replayed) form reads x_host anew per call
            plan = sb.GemvHostPlan(w, x_host, x_dev, y_dev, y_host)
            x2 = synth.gen_x(202, 1, k)[0]
            x_host.copy_(t.from_numpy(x2.view(np.float16).copy()))
            y_host.zero_()
            plan()
            t.cuda.synchronize()
            y2_dev = t.empty(n, dtype=t.float16, device="cuda")
            sb.bonsai_gemv(w, dev(x2), y2_dev)
            assert sb.bonsai_check_async() == 0
            assert np.array_equal(y_host.numpy().view(np.uint16), host(y2_dev))


# ------------------------------------------ gated feed-forward (SwiGLU)
SWIGLU_CASES = [(BIN, 8, 128, 1), (TER, 8, 128, 1), (BIN, 24, 640, 3), (TER, 40, 640, 5),
                (TER, 56, 1152, 8), (BIN, 200, 1024, 9), (TER, 136, 1024, 300),
                (BIN, 64, 256, 257)]


@pytest.mark.parametrize("fmt,f,k,m", SWIGLU_CASES)
def test_swiglu_full(fmt, f, k, m):
    """Every output of h = silu(g) * u for the interleaved gate/up matrix:
    decode kernel (m <= 8, ternary m > 4 in two launches) and GEMM (m > 8,
    ragged feature and token tiles)."""
    t = torch()
    w, packed, scales = weights(fmt, 150 + f, 2 * f, k)
    x = synth.gen_x(151 + m, m, k)
    h = Guarded((m, f), t.float16)
    sb.bonsai_gemm_swiglu(w, dev(x), h.t)
    assert sb.bonsai_check_async() == 0
    href, g, u, ng, nu = oracle.swiglu(fmt, packed, scales, x)
    assert_swiglu_close(host(h.t), href, g, u, ng, nu, "swiglu fmt=%d f=%d k=%d m=%d" % (fmt, f, k, m))
    h.check()


@pytest.mark.parametrize("fmt,m", [(BIN, 1), (TER, 1), (TER, 8), (BIN, 100), (BIN, 512), (TER, 512)])
def test_swiglu_workload(fmt, m):
    """Gate/up of the 64-layer model (F=17408, K=5120), sampled features."""
    t = torch()
    f, k = 17408, 5120
    w, packed, scales = weights(fmt, 160 + fmt, 2 * f, k)
    x = synth.gen_x(161 + m, m, k)
    h = Guarded((m, f), t.float16)
    sb.bonsai_gemm_swiglu(w, dev(x), h.t)
    assert sb.bonsai_check_async() == 0
    fs = sample_idx(f, [0, 7, 8, 63, 64, 127, 128, f - 9, f - 8, f - 1], 50, 7)
    ms = sample_idx(m, [0, m - 1], 12, 8)
    href, g, u, ng, nu = oracle.swiglu(fmt, packed, scales, x, f_sel=fs, m_sel=ms)
    assert_swiglu_close(host(h.t)[np.ix_(ms, fs)], href, g, u, ng, nu, "swiglu workload m=%d" % m)
    h.check()


def test_swiglu_zero_gate_rows():
    """Ternary gate rows that are all zero give h = +-0 exactly, whatever u."""
    t = torch()
    f, k = 16, 640
    codes = synth.gen_ternary_codes(170, 2 * f, k)
    codes[0:8] = 0          # gate rows of features 0..7
    codes[24:32] = 0        # up rows of features 8..15
    rb = sb.bonsai_packed_row_bytes(TER, k)
    packed_gpu = t.empty((2 * f, rb), dtype=t.uint8, device="cuda")
    sb.bonsai_pack_ternary(dev(codes), packed_gpu)
    scales = synth.gen_scales(171, 2 * f, k)
    w = sb.Weights(TER, 2 * f, k, packed_gpu, dev(scales))
    for m in (1, 3, 20):
        x = synth.gen_x(172 + m, m, k)
        h = t.empty((m, f), dtype=t.float16, device="cuda")
        sb.bonsai_gemm_swiglu(w, dev(x), h)
        assert sb.bonsai_check_async() == 0
        hv = host(h)
        assert np.all((hv & 0x7FFF) == 0), m
        href, g, u, ng, nu = oracle.swiglu(TER, oracle.pack_ternary(codes), scales, x)
        assert np.all(href == 0.0)
        assert_swiglu_close(hv, href, g, u, ng, nu, "zero rows m=%d" % m)


# --------------------------------------------- activation binarisation
def scale_tol(ref, k):
    """Bound on |a_s_gpu - mean|x|| for the FP16 scale: the FP32 sum of k
    non-negative terms and the division are within (k + 1) * 2^-24 of the
    exact mean, relative; the FP16 rounding adds half an ulp (2^-11 relative,
    2^-25 absolute in the subnormal range)."""
    return (2.0 ** -11 + (k + 2) * 2.0 ** -24) * np.abs(ref) + 2.0 ** -25


def check_binarized(bits_gpu, as_gpu, x, what):
    k = x.shape[1]
    bits_ref, as_ref = oracle.binarize(x)
    assert np.array_equal(bits_gpu.view(np.uint32), bits_ref), what + ": codes"
    got = as_gpu.view(np.float16).astype(np.float64)
    nan = np.isnan(as_ref)
    assert np.array_equal(np.isnan(got), nan), what + ": NaN scales"
    g, r = got[~nan], as_ref[~nan]
    inf = np.isinf(r)
    assert np.array_equal(g[inf], r[inf]), what + ": infinite scales"
    err = np.abs(g[~inf] - r[~inf])
    assert np.all(err <= scale_tol(r[~inf], k)), (what, float(err.max(initial=0.0)))


@pytest.mark.parametrize("m,k", [(1, 128), (3, 640), (5, 4096), (512, 4096), (1, 17408),
                                 (7, 5120), (1300, 256), (2, 1152), (4096, 4096),
                                 (2500, 640), (10000, 128)])
def test_binarize_rows(m, k):
    t = torch()
    x = synth.gen_x(130 + m, m, k)
    bits = Guarded((m, k // 32), t.int32)
    a_s = Guarded((m,), t.float16)
    sb.bonsai_binarize_activations(dev(x), bits.t, a_s.t)
    assert sb.bonsai_check_async() == 0
    check_binarized(host(bits.t), host(a_s.t), x, "binarize m=%d k=%d" % (m, k))
    bits.check()
    a_s.check()


def test_binarize_special_values():
    """Both zeros give +1, a NaN gives -1 and a NaN scale, infinities keep
    their sign and give an infinite scale, subnormals keep theirs."""
    t = torch()
    k = 256
    f = np.float16
    rows = np.zeros((8, k), dtype=np.float16)
    rows[1] = f(-0.0)
    rows[2] = np.where(np.arange(k) % 2, f(-0.0), f(0.0))
    rows[3] = f(1.0)
    rows[3, 77] = f(np.nan)
    rows[4] = f(-1.0)
    rows[4, 3] = -f(np.nan)
    rows[5] = np.where(np.arange(k) % 3, f(np.inf), f(-np.inf))
    rows[6] = np.where(np.arange(k) % 2, f(6e-8), f(-6e-8))  # smallest subnormal
    rows[7] = np.where(np.arange(k) < 200, f(65504.0), f(-65504.0))  # largest finite
    x = rows.view(np.uint16)
    bits = t.empty((8, k // 32), dtype=t.int32, device="cuda")
    a_s = t.empty(8, dtype=t.float16, device="cuda")
    sb.bonsai_binarize_activations(dev(x), bits, a_s)
    assert sb.bonsai_check_async() == 0
    check_binarized(host(bits), host(a_s), x, "special values")


def test_xnor_from_fp16_activations():
    """FP16 activations -> bonsai_binarize_activations -> bonsai_xnor_gemm,
    against the oracle's binarisation composed with its XNOR product (unit
    activation scale, then times the exact mean |x|). D is exact; Y carries
    the scale's FP16 rounding, inside 2e-3 of sum a_s*128*|s_g|."""
    t = torch()
    for (m, n, k) in ((37, 200, 1024), (512, 4096, 4096)):
        x = synth.gen_x(140 + m, m, k)
        w_bits = synth.gen_binary_words(141 + m, n, k)
        s = synth.gen_scales(142 + m, n, k)
        w = sb.Weights(BIN, n, k, dev(w_bits.view(np.uint8).reshape(n, -1)), dev(s))
        bits = t.empty((m, k // 32), dtype=t.int32, device="cuda")
        a_s = t.empty(m, dtype=t.float16, device="cuda")
        d = Guarded((m, n), t.int32)
        y = Guarded((m, n), t.float16)
        sb.bonsai_binarize_activations(dev(x), bits, a_s)
        sb.bonsai_xnor_gemm(bits, a_s, w, d.t, y.t)
        assert sb.bonsai_check_async() == 0
        bits_ref, as_ref = oracle.binarize(x)
        ms = sample_idx(m, [0, m - 1], 20, 5)
        ns = sample_idx(n, [0, 63, 64, n - 1], 30, 6)
        unit = np.full(m, np.float16(1.0).view(np.uint16), dtype=np.uint16)
        d_ref, y1, n1 = oracle.xnor(bits_ref, unit, w_bits, s, k, n_sel=ns, m_sel=ms)
        assert np.array_equal(host(d.t)[np.ix_(ms, ns)].astype(np.int64), d_ref)
        sc = as_ref[ms][:, None]
        assert_close(host(y.t)[np.ix_(ms, ns)], sc * y1, sc * n1, "xnor from fp16 m=%d" % m)
        d.check()
        y.check()


# ------------------------------------------------- signed Hadamard rotation
def hadamard_bound(ref, x, block):
    """FP32 butterflies: each of the log2(block) stages rounds a partial sum
    bounded by the block's sum |x|, and the 1/sqrt(block) constant and product
    round once more each; the FP16 store adds half an ulp of the result
    (2^-11 relative, 2^-25 absolute for subnormals)."""
    m, k = x.shape
    s = np.abs(x.view(np.float16).astype(np.float64)).reshape(m, k // block, block).sum(axis=2)
    s = np.repeat(s, block, axis=1) / np.sqrt(block)
    e = (np.log2(block) + 3) * 2.0 ** -24 * s
    return e + 2.0 ** -11 * (np.abs(ref) + e) + 2.0 ** -25


HADAMARD_CASES = [(1, 128, 128, False), (3, 640, 128, True), (5, 5120, 128, True),
                  (2, 5120, 1024, True), (4, 17408, 512, True), (7, 1024, 256, True),
                  (3, 256, 8, True), (2, 384, 32, True), (1, 2048, 64, False),
                  (512, 5120, 128, True), (33, 17408, 1024, False)]


@pytest.mark.parametrize("m,k,block,signed", HADAMARD_CASES)
def test_hadamard(m, k, block, signed):
    t = torch()
    x = synth.gen_x(190 + m, m, k)
    bits = synth.gen_binary_words(191 + k, 1, k)[0] if signed else None
    out = Guarded((m, k), t.float16)
    sb.bonsai_hadamard(dev(x), out.t, block, None if bits is None else dev(bits.view(np.int32)))
    assert sb.bonsai_check_async() == 0
    ref = oracle.hadamard(x, block, bits)
    bad, first, worst = oracle.compare_f16(host(out.t), ref, hadamard_bound(ref, x, block), 1.0)
    assert bad == 0, ("hadamard", m, k, block, bad, first, worst)
    out.check()


def test_hadamard_in_place_and_involution():
    """In place gives the same bits as out of place; with all signs +1 and an
    even log2(block), rotating twice returns x up to the two roundings."""
    t = torch()
    m, k = 6, 4096
    x = synth.gen_x(195, m, k)
    for block in (256, 1024):
        a = dev(x)
        b = t.empty_like(a)
        sb.bonsai_hadamard(a, b, block)
        sb.bonsai_hadamard(a, a, block)
        assert sb.bonsai_check_async() == 0
        assert np.array_equal(host(a), host(b))
        back = t.empty_like(a)
        sb.bonsai_hadamard(a, back, block)
        assert sb.bonsai_check_async() == 0
        xv = x.view(np.float16).astype(np.float64)
        err = np.abs(host(back).view(np.float16).astype(np.float64) - xv)
        assert np.all(err <= 4 * 2.0 ** -11 * np.sqrt(np.mean(xv ** 2)) + 2.0 ** -11 * np.abs(xv))


# ------------------------------------------------------- failure detection
def test_bounded_wait_reports_timeout_and_device_stays_usable():
    """A wait that nothing completes gives up after its limit: the status
    word reads BONSAI_ERR_TIMEOUT once, then clears, and products still run."""
    t = torch()
    t0 = __import__("time").perf_counter()
    sb.bonsai_selftest_wait_timeout(2_000_000)  # 2 ms
    st = sb.bonsai_check_async()
    elapsed = __import__("time").perf_counter() - t0
    assert sb.STATUS[st] == "BONSAI_ERR_TIMEOUT"
    assert elapsed < 5.0
    assert sb.bonsai_check_async() == 0  # cleared
    w, packed, scales = weights(TER, 5, 64, 640)
    x = synth.gen_x(7, 1, 640)
    y = t.empty(64, dtype=t.float16, device="cuda")
    sb.bonsai_gemv(w, dev(x[0]), y)
    assert sb.bonsai_check_async() == 0
    y_ref, nrm = oracle.linear(TER, packed, scales, x)
    assert_close(host(y), y_ref[0], nrm[0], "after a timeout")


# ------------------------------------------------------------ graph capture
def test_graph_capture_matches_eager():
    """Launches captured into a CUDA graph (programmatic dependent launch
    edges included) give the same bits as eager launches."""
    t = torch()
    wb, _, _ = weights(BIN, 5, 640, 1024, flags=sb.BONSAI_WEIGHTS_PREFETCH)
    wt, _, _ = weights(TER, 6, 900, 5120, flags=sb.BONSAI_WEIGHTS_PREFETCH)
    x1 = dev(synth.gen_x(1, 1, 1024)[0])
    x2 = dev(synth.gen_x(2, 1, 5120)[0])
    xm = dev(synth.gen_x(3, 300, 5120))

    def run(ys):
        sb.bonsai_gemv(wb, x1, ys[0])
        sb.bonsai_gemv(wt, x2, ys[1])
        sb.bonsai_gemm(wt, xm, ys[2])
        sb.bonsai_gemv(wb, x1, ys[3])

    def bufs():
        return [t.empty(640, dtype=t.float16, device="cuda"),
                t.empty(900, dtype=t.float16, device="cuda"),
                t.empty((300, 900), dtype=t.float16, device="cuda"),
                t.empty(640, dtype=t.float16, device="cuda")]
    eager, graphed = bufs(), bufs()
    run(eager)
    t.cuda.synchronize()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g):
        run(graphed)
    for _ in range(3):
        g.replay()
    assert sb.bonsai_check_async() == 0
    for a, b in zip(eager, graphed):
        assert t.equal(a.view(t.int16), b.view(t.int16))


def test_graph_capture_chained_newer_entry_points():
    """The later entry points captured into one CUDA graph, each consuming the
    previous one's output (as in a decode layer): Hadamard rotation -> gated
    feed-forward (decode and tensor-core paths) -> down product, and FP16
    binarisation -> XNOR. Replays give the bits of eager calls."""
    t = torch()
    k, f = 1024, 256
    wgu, _, _ = weights(TER, 40, 2 * f, k, flags=sb.BONSAI_WEIGHTS_PREFETCH)
    wdown, _, _ = weights(BIN, 41, 320, f)
    wx = sb.Weights(BIN, 384, k, dev(synth.gen_binary_words(42, 384, k).view(np.uint8).reshape(384, -1)),
                    dev(synth.gen_scales(43, 384, k)))
    signs = dev(synth.gen_binary_words(44, 1, k)[0].view(np.int32))
    x1 = dev(synth.gen_x(45, 1, k))
    xm = dev(synth.gen_x(46, 300, k))

    def bufs():
        return {"r1": t.empty((1, k), dtype=t.float16, device="cuda"),
                "rm": t.empty((300, k), dtype=t.float16, device="cuda"),
                "h1": t.empty((1, f), dtype=t.float16, device="cuda"),
                "hm": t.empty((300, f), dtype=t.float16, device="cuda"),
                "y1": t.empty((1, 320), dtype=t.float16, device="cuda"),
                "ym": t.empty((300, 320), dtype=t.float16, device="cuda"),
                "bits": t.empty((300, k // 32), dtype=t.int32, device="cuda"),
                "as": t.empty(300, dtype=t.float16, device="cuda"),
                "d": t.empty((300, 384), dtype=t.int32, device="cuda"),
                "yx": t.empty((300, 384), dtype=t.float16, device="cuda")}

    def run(b):
        sb.bonsai_hadamard(x1, b["r1"], 128, signs)
        sb.bonsai_hadamard(xm, b["rm"], 256, signs)
        sb.bonsai_gemm_swiglu(wgu, b["r1"], b["h1"])
        sb.bonsai_gemm_swiglu(wgu, b["rm"], b["hm"])
        sb.bonsai_gemm(wdown, b["h1"], b["y1"])
        sb.bonsai_gemm(wdown, b["hm"], b["ym"])
        sb.bonsai_binarize_activations(b["rm"], b["bits"], b["as"])
        sb.bonsai_xnor_gemm(b["bits"], b["as"], wx, b["d"], b["yx"])

    eager, graphed = bufs(), bufs()
    run(eager)
    t.cuda.synchronize()
    assert sb.bonsai_check_async() == 0
    s = t.cuda.Stream()
    s.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(s):
        run(graphed)  # eager once on the capture stream: one-time set-up outside the capture
    t.cuda.current_stream().wait_stream(s)
    t.cuda.synchronize()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g):
        run(graphed)
    for _ in range(3):
        g.replay()
    assert sb.bonsai_check_async() == 0
    for name in eager:
        a, b = eager[name], graphed[name]
        assert t.equal(a.view(t.int16) if a.dtype == t.float16 else a,
                       b.view(t.int16) if b.dtype == t.float16 else b), name
