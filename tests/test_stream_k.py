"""Stream-K schedule of the tensor-core GEMM (bonsai_gemm_ws,
bonsai_gemm_swiglu_ws) against the oracle and against the plain schedule
(needs a GPU).

Shapes whose 128 x 256 tiles leave a last wave short of the SMs: the N=5120
products of a pp512 layer (80 tiles), whole waves plus a cut tail (160
tiles), and few tiles cut into many ranges (one finishing range adding nine
partial tiles)."""
import numpy as np
import pytest

import oracle
import sub_bit_weight_binary_b300 as sb
from sub_bit_weight_binary_b300 import synth
from gpu_util import TOL, Guarded, assert_close, assert_swiglu_close, dev, host, torch, weights

pytestmark = pytest.mark.gpu
BIN, TER = sb.BONSAI_FMT_BINARY, sb.BONSAI_FMT_TERNARY


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch().cuda.is_available():
        pytest.skip("no CUDA device")
    sb.lib()
    oracle.lib()
    yield
    assert sb.bonsai_check_async() == 0


def sample_idx(total, edges, count, seed):
    rng = np.random.default_rng(seed)
    idx = set(int(e) for e in edges if 0 <= e < total)
    idx.update(int(v) for v in rng.integers(0, total, count))
    return np.array(sorted(idx), dtype=np.int64)


def tile_edges(total, step):
    """First, second and last index of every tile of `step`, plus the end."""
    e = []
    for t0 in range(0, total, step):
        e += [t0, t0 + 1, t0 + step - 1]
    return e + [total - 1]


def sms():
    return torch().cuda.get_device_properties(0).multi_processor_count


def counters(ws, m, n):
    """The workspace's counter words, one per cut tile (128 x 256 tiles of the
    last, partial wave); all zero after a completed call."""
    tiles = ((n + 127) // 128) * ((m + 255) // 256)
    cut = tiles % sms()
    return host(ws[: 4 * cut].view(torch().int32)).astype(np.int64)


@pytest.mark.parametrize("fmt,m,n,k", [(BIN, 300, 1000, 1280), (TER, 300, 1000, 1280),
                                       (TER, 20, 640, 5120), (BIN, 20, 640, 5120)])
def test_stream_k_full(fmt, m, n, k):
    """Every output against the oracle; the workspace's counters are zero
    again afterwards and a second call gives bit-identical y."""
    t = torch()
    w, packed, scales = weights(fmt, 200 + m, n, k)
    x = synth.gen_x(201 + n % 17, m, k)
    ws = sb.gemm_workspace(w, m)
    assert ws is not None, "this shape should take the stream-K schedule"
    y1 = Guarded((m, n), t.float16)
    y2 = Guarded((m, n), t.float16)
    sb.bonsai_gemm_ws(w, dev(x), y1.t, ws)
    assert sb.bonsai_check_async() == 0
    assert counters(ws, m, n).max() == 0
    sb.bonsai_gemm_ws(w, dev(x), y2.t, ws)
    assert sb.bonsai_check_async() == 0
    assert t.equal(y1.t.view(t.int16), y2.t.view(t.int16))
    y_ref, nrm = oracle.linear(fmt, packed, scales, x)
    assert_close(host(y1.t), y_ref, nrm, "stream-K fmt=%d m=%d n=%d k=%d" % (fmt, m, n, k))
    y1.check()
    y2.check()


@pytest.mark.parametrize("fmt", [BIN, TER])
def test_stream_k_whole_waves_and_tail(fmt):
    """160 tiles: one whole wave (148 SMs), the last 12 tiles cut into ranges;
    all tokens, sampled features with every tile edge."""
    t = torch()
    m, n, k = 100, 20480, 1280
    w, packed, scales = weights(fmt, 210, n, k)
    x = synth.gen_x(211, m, k)
    ws = sb.gemm_workspace(w, m)
    assert ws is not None
    y = Guarded((m, n), t.float16)
    sb.bonsai_gemm_ws(w, dev(x), y.t, ws)
    assert sb.bonsai_check_async() == 0
    assert counters(ws, m, n).max() == 0
    whole = (n // 128) // sms() * sms() * 128  # rows of the whole wave
    ns = sample_idx(n, tile_edges(n, 128)[::7] + list(range(whole - 2, n)), 200, 3)
    y_ref, nrm = oracle.linear(fmt, packed, scales, x, n_sel=ns)
    assert_close(host(y.t)[:, ns], y_ref, nrm, "stream-K tail fmt=%d" % fmt)
    y.check()


@pytest.mark.parametrize("fmt", [BIN, TER])
@pytest.mark.parametrize("k", [5120, 17408])
def test_stream_k_prefill_small_n(fmt, k):
    """The o (K=5120) and down (K=17408) products of a pp512 layer, N=5120:
    every tile edge row and column plus samples, against the oracle; and the
    plain schedule agrees within the sum of the two bounds."""
    t = torch()
    m, n = 512, 5120
    w, packed, scales = weights(fmt, 220 + k % 7, n, k)
    x = synth.gen_x(221, m, k)
    ws = sb.gemm_workspace(w, m)
    assert ws is not None
    y = Guarded((m, n), t.float16)
    sb.bonsai_gemm_ws(w, dev(x), y.t, ws)
    y0 = t.empty((m, n), dtype=t.float16, device="cuda")
    sb.bonsai_gemm(w, dev(x), y0)
    assert sb.bonsai_check_async() == 0
    assert counters(ws, m, n).max() == 0
    ms = sample_idx(m, [0, 1, 255, 256, 257, m - 1], 24, 4)
    ns = sample_idx(n, tile_edges(n, 128), 40, 5)
    y_ref, nrm = oracle.linear(fmt, packed, scales, x, n_sel=ns, m_sel=ms)
    got = host(y.t)[np.ix_(ms, ns)]
    assert_close(got, y_ref, nrm, "stream-K pp512 fmt=%d k=%d" % (fmt, k))
    a = got.view(np.float16).astype(np.float64)
    b = host(y0)[np.ix_(ms, ns)].view(np.float16).astype(np.float64)
    assert np.all(np.abs(a - b) <= 2 * TOL * nrm + 1e-30)
    y.check()


@pytest.mark.parametrize("fmt", [BIN, TER])
def test_stream_k_swiglu(fmt):
    """Gated feed-forward with the stream-K schedule: F=2560 (80 tiles at
    512 tokens), every output of sampled tokens."""
    t = torch()
    m, f, k = 512, 2560, 1280
    w, packed, scales = weights(fmt, 230, 2 * f, k)
    x = synth.gen_x(231, m, k)
    ws = sb.gemm_workspace(w, m)
    assert ws is not None
    h = Guarded((m, f), t.float16)
    sb.bonsai_gemm_swiglu_ws(w, dev(x), h.t, ws)
    assert sb.bonsai_check_async() == 0
    assert counters(ws, m, 2 * f).max() == 0
    ms = sample_idx(m, [0, 255, 256, m - 1], 20, 6)
    href, g, u, ng, nu = oracle.swiglu(fmt, packed, scales, x, m_sel=ms)
    assert_swiglu_close(host(h.t)[ms], href, g, u, ng, nu, "stream-K swiglu fmt=%d" % fmt)
    h.check()


def test_stream_k_small_workspace_runs_plain():
    """A workspace below the reported size (or none) runs the plain schedule."""
    t = torch()
    m, n, k = 300, 1000, 1280
    w, packed, scales = weights(TER, 240, n, k)
    x = synth.gen_x(241, m, k)
    need = sb.bonsai_gemm_workspace_bytes(w, m)
    assert need > 0
    small = t.zeros(need - 256, dtype=t.uint8, device="cuda")
    y1 = t.empty((m, n), dtype=t.float16, device="cuda")
    y2 = t.empty((m, n), dtype=t.float16, device="cuda")
    sb.bonsai_gemm_ws(w, dev(x), y1, small)
    sb.bonsai_gemm(w, dev(x), y2)
    assert sb.bonsai_check_async() == 0
    assert t.equal(y1.view(t.int16), y2.view(t.int16))
    assert int(small.count_nonzero()) == 0


def test_stream_k_rejects_unaligned_workspace():
    t = torch()
    m, n, k = 300, 1000, 1280
    w, _, _ = weights(TER, 242, n, k)
    x = dev(synth.gen_x(243, m, k))
    need = sb.bonsai_gemm_workspace_bytes(w, m)
    buf = t.zeros(need + 512, dtype=t.uint8, device="cuda")
    y = t.empty((m, n), dtype=t.float16, device="cuda")
    with pytest.raises(sb.BonsaiError) as e:
        sb.bonsai_gemm_ws(w, x, y, buf[16:])
    assert "BONSAI_ERR_ALIGN" in str(e.value)


def test_stream_k_not_taken_when_tiles_fill_the_sms():
    """A product whose tiles fill the SMs in whole waves needs no workspace."""
    w, _, _ = weights(TER, 244, 128 * sms(), 640)
    assert sb.bonsai_gemm_workspace_bytes(w, 256) == 0
