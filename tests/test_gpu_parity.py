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
from gpu_util import Guarded, assert_close, dev, host, torch, weights

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
    (TER, 17408, 5120),   # ternary decode workload (M=1, K=5120, N=17408)
    (TER, 1, 128), (TER, 17, 640), (TER, 33, 5120), (TER, 40, 17408),
    (TER, 5120, 17408), (TER, 300, 1280), (TER, 129, 384),
    # the decode sweep's stacked q/k/v and gate/up matrices
    (BIN, 15360, 5120), (TER, 15360, 5120), (BIN, 34816, 5120), (TER, 34816, 5120),
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
@pytest.mark.parametrize("m,n,k", [(2, 300, 1024), (5, 1024, 5120), (8, 129, 640), (3, 64, 17408)])
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
                                   (257, 130, 5120), (256, 256, 320 * 4)])
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
@pytest.mark.parametrize("m,n,k", [(64, 256, 4096), (70, 100, 640), (1, 1, 128), (130, 65, 1024)])
def test_xnor_full(m, n, k):
    t = torch()
    a_bits, a_s, w_bits, s = synth.gen_xnor_inputs(90 + m, m, n, k)
    w = sb.Weights(BIN, n, k, dev(w_bits.view(np.uint8).reshape(n, -1)), dev(s))
    d = Guarded((m, n), t.int32)
    y = Guarded((m, n), t.float16)
    sb.bonsai_xnor_gemm(dev(a_bits.view(np.int32)), dev(a_s), w, d.t, y.t)
    assert sb.bonsai_check_async() == 0
    d_ref, y_ref, nrm = oracle.xnor(a_bits, a_s, w_bits, s, k)
    assert np.array_equal(host(d.t).astype(np.int64), d_ref)
    assert_close(host(y.t), y_ref, nrm, "xnor")
    d.check()
    y.check()


def test_xnor_workload():
    """XNOR workload M=512, K=4096, N=4096: D sampled against the oracle and
    every D checked against the popcount route of numpy; Y sampled."""
    t = torch()
    m, n, k = 512, 4096, 4096
    a_bits, a_s, w_bits, s = synth.gen_xnor_inputs(95, m, n, k)
    w = sb.Weights(BIN, n, k, dev(w_bits.view(np.uint8).reshape(n, -1)), dev(s))
    d = Guarded((m, n), t.int32)
    y = Guarded((m, n), t.float16)
    sb.bonsai_xnor_gemm(dev(a_bits.view(np.int32)), dev(a_s), w, d.t, y.t)
    d_only = t.empty((m, n), dtype=t.int32, device="cuda")
    sb.bonsai_xnor_gemm(dev(a_bits.view(np.int32)), dev(a_s), w, d_only, None)
    y_only = t.empty((m, n), dtype=t.float16, device="cuda")
    sb.bonsai_xnor_gemm(dev(a_bits.view(np.int32)), dev(a_s), w, None, y_only)
    assert sb.bonsai_check_async() == 0
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
