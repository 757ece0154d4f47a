"""One-token binary and ternary products on the per-position table kernels
(bonsai_gemv_ws, bonsai_gemv_host_ws, bonsai_gemm_ws / bonsai_gemm_swiglu_ws
with m = 1) against the oracle (needs a GPU).

Shapes: the decode products of the pages' 27B decoder (N=17408 x K=5120, the
down product N=5120 x K=17408 with a partial last 640-code slice), K=1024
and K=3072 (partial last slice, ragged last chunk of rows, a last stage of
4 rows), rows with few or no nonzero codes, activations over many binades,
and the gated feed-forward epilogue; binary at the same decode shapes and
K=1024 / 3072. The kernels take products with at least 768 (ternary) or 640
(binary) rows per thread block, hence the row counts."""
import numpy as np
import pytest

import oracle
import sub_bit_weight_binary_b300 as sb
from sub_bit_weight_binary_b300 import synth
from gpu_util import (TOL, Guarded, assert_close, assert_swiglu_close, dev, host, torch,
                      weights)

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


def sms():
    return torch().cuda.get_device_properties(0).multi_processor_count


def counters(ws, n, k, fmt=None):
    """The workspace's arrival counters (after the partial sums): all zero
    after a completed call. Layout: slices of 640 (ternary) or 1024 (binary)
    codes, chunks of rc rows."""
    s = -(-k // (1024 if fmt == BIN else 640))
    c0 = sms() // s
    rc = -(-(-(-n // c0)) // 16) * 16
    c = -(-n // rc)
    off = c * s * rc * 4
    return host(ws[off: off + 4 * c * s].view(torch().int32))


def f16(y_u16):
    return y_u16.view(np.float16).astype(np.float64)


def ternary_from_codes(codes, seed):
    t = torch()
    n, k = codes.shape
    rb = sb.bonsai_packed_row_bytes(TER, k)
    packed_gpu = t.empty((n, rb), dtype=t.uint8, device="cuda")
    sb.bonsai_pack_ternary(dev(codes), packed_gpu)
    scales = synth.gen_scales(seed, n, k)
    return sb.Weights(TER, n, k, packed_gpu, dev(scales)), oracle.pack_ternary(codes), scales


@pytest.mark.parametrize("fmt,n,k", [(TER, 17408, 5120), (TER, 5120, 17408), (TER, 57000, 1024),
                                     (TER, 22300, 3072), (BIN, 20000, 5120), (BIN, 5120, 17408),
                                     (BIN, 95000, 1024), (BIN, 40000, 3072)])
def test_lut_full(fmt, n, k):
    """Every output against the oracle; a second call is bit-identical and
    the counters are zero again after each call."""
    t = torch()
    w, packed, scales = weights(fmt, 300 + k % 11, n, k)
    x = synth.gen_x(301 + n % 7, 1, k)
    ws = sb.gemv_workspace(w)
    assert ws is not None, "this shape should take the table kernel"
    y1 = Guarded((n,), t.float16)
    y2 = Guarded((n,), t.float16)
    sb.bonsai_gemv_ws(w, dev(x[0]), y1.t, ws)
    assert sb.bonsai_check_async() == 0
    assert counters(ws, n, k, fmt).max() == 0
    sb.bonsai_gemv_ws(w, dev(x[0]), y2.t, ws)
    assert sb.bonsai_check_async() == 0
    assert counters(ws, n, k, fmt).max() == 0
    assert t.equal(y1.t.view(t.int16), y2.t.view(t.int16))
    y_ref, nrm = oracle.linear(fmt, packed, scales, x)
    assert_close(host(y1.t), y_ref[0], nrm[0], "table kernel fmt=%d n=%d k=%d" % (fmt, n, k))
    y1.check()
    y2.check()


@pytest.mark.parametrize("fmt", [BIN, TER])
def test_lut_agrees_with_streaming_kernel(fmt):
    """The table kernel and bonsai_gemv's kernel each meet the bound, so they
    agree within twice it."""
    t = torch()
    n, k = 20000 if fmt == BIN else 17408, 5120
    w, packed, scales = weights(fmt, 310, n, k)
    x = dev(synth.gen_x(311, 1, k)[0])
    ws = sb.gemv_workspace(w)
    y0 = t.empty(n, dtype=t.float16, device="cuda")
    y1 = t.empty(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv(w, x, y0)
    sb.bonsai_gemv_ws(w, x, y1, ws)
    assert sb.bonsai_check_async() == 0
    _, nrm = oracle.linear(fmt, packed, scales, host(x)[None, :], n_sel=np.arange(0, n, 7))
    a = f16(host(y0))[::7]
    b = f16(host(y1))[::7]
    assert np.all(np.abs(a - b) <= 2 * TOL * nrm[0] + 1e-30)


@pytest.mark.parametrize("per_mille", [20, 0])
def test_lut_sparse_and_zero_rows(per_mille):
    """Rows with few (or no) nonzero codes meet the bound against their own
    small norm; all-zero rows give exactly zero."""
    n, k = 14000, 5120
    codes = np.empty((n, k), dtype=np.int8)
    for r0 in range(0, n, 1000):  # in row blocks: bounded host memory
        rows = min(1000, n - r0)
        wr = synth.words(320 + per_mille, 0x51, r0 * k, rows * k)
        keep = (wr >> np.uint64(54)) < np.uint64(per_mille * 1024 // 1000)
        codes[r0:r0 + rows] = np.where(keep, np.where((wr & np.uint64(1)) == 1, 1, -1),
                                       0).astype(np.int8).reshape(rows, k)
    codes[::5] = 0  # every fifth row all zero
    w, packed, scales = ternary_from_codes(codes, 321)
    ws = sb.gemv_workspace(w)
    assert ws is not None
    x = synth.gen_x(322, 1, k)
    y = Guarded((n,), torch().float16)
    sb.bonsai_gemv_ws(w, dev(x[0]), y.t, ws)
    assert sb.bonsai_check_async() == 0
    y_ref, nrm = oracle.linear(TER, packed, scales, x)
    got = host(y.t)
    assert_close(got, y_ref[0], nrm[0], "table kernel sparse %d/1000" % per_mille)
    assert np.all(f16(got)[::5] == 0.0)
    y.check()


@pytest.mark.parametrize("fmt", [BIN, TER])
def test_lut_wide_range_activations(fmt):
    """x over seven binades, both signs, one tenth exact zeros."""
    n, k = 20000 if fmt == BIN else 17408, 5120
    w, packed, scales = weights(fmt, 330, n, k)
    rng = np.random.default_rng(331)
    mag = 10.0 ** rng.uniform(-4, 3, size=k)
    xv = (mag * rng.choice([-1.0, 1.0], size=k)).astype(np.float16)
    xv[rng.integers(0, k, size=k // 10)] = 0
    x = xv.view(np.uint16)[None, :]
    ws = sb.gemv_workspace(w)
    assert ws is not None
    y = Guarded((n,), torch().float16)
    sb.bonsai_gemv_ws(w, dev(x[0]), y.t, ws)
    assert sb.bonsai_check_async() == 0
    y_ref, nrm = oracle.linear(fmt, packed, scales, x)
    assert_close(host(y.t), y_ref[0], nrm[0], "table kernel wide-range x fmt=%d" % fmt)
    y.check()


@pytest.mark.parametrize("fmt", [BIN, TER])
def test_lut_swiglu(fmt):
    """Gated feed-forward input of one token (F=8704 ternary / 10240 binary
    features from 2F interleaved rows): every h against the oracle's
    silu(g)*u bound."""
    t = torch()
    f, k = 10240 if fmt == BIN else 8704, 5120
    w, packed, scales = weights(fmt, 340, 2 * f, k)
    x = synth.gen_x(341, 1, k)
    ws = sb.gemv_workspace(w)
    assert ws is not None
    assert sb.bonsai_gemm_workspace_bytes(w, 1) == ws.numel()
    h = Guarded((1, f), t.float16)
    sb.bonsai_gemm_swiglu_ws(w, dev(x), h.t, ws)
    assert sb.bonsai_check_async() == 0
    assert counters(ws, 2 * f, k, fmt).max() == 0
    href, g, u, ng, nu = oracle.swiglu(fmt, packed, scales, x)
    assert_swiglu_close(host(h.t), href, g, u, ng, nu, "table kernel swiglu fmt=%d" % fmt)
    h.check()


def test_lut_gemm_ws_one_token_is_the_same_kernel():
    t = torch()
    n, k = 22300, 3072
    w, _, _ = weights(TER, 350, n, k)
    x = dev(synth.gen_x(351, 1, k))
    ws = sb.gemv_workspace(w)
    y1 = t.empty(n, dtype=t.float16, device="cuda")
    y2 = t.empty((1, n), dtype=t.float16, device="cuda")
    sb.bonsai_gemv_ws(w, x[0], y1, ws)
    sb.bonsai_gemm_ws(w, x, y2, ws)
    assert sb.bonsai_check_async() == 0
    assert t.equal(y1.view(t.int16), y2[0].view(t.int16))


def test_lut_host_buffers_and_prefetch_flag():
    """bonsai_gemv_host with the workspace (pinned x in, y out) and weights
    flagged for early streaming give the device call's y bit for bit."""
    t = torch()
    n, k = 17408, 5120
    w, _, _ = weights(TER, 360, n, k)
    wp, _, _ = weights(TER, 360, n, k, flags=sb.BONSAI_WEIGHTS_PREFETCH)
    xh = t.from_numpy(synth.gen_x(361, 1, k)[0].view(np.float16)).pin_memory()
    xd = xh.cuda()
    ws = sb.gemv_workspace(w)
    y_dev = t.empty(n, dtype=t.float16, device="cuda")
    y_ref = t.empty(n, dtype=t.float16, device="cuda")
    y_pf = t.empty(n, dtype=t.float16, device="cuda")
    y_host = t.empty(n, dtype=t.float16).pin_memory()
    x_dev = t.empty(k, dtype=t.float16, device="cuda")
    sb.bonsai_gemv_ws(w, xd, y_ref, ws)
    sb.bonsai_gemv_ws(wp, xd, y_pf, ws)
    sb.bonsai_gemv_host(w, xh, x_dev, y_dev, y_host, workspace=ws)
    assert sb.bonsai_check_async() == 0
    assert t.equal(y_pf.view(t.int16), y_ref.view(t.int16))
    assert t.equal(y_host.view(t.int16), y_ref.cpu().view(t.int16))


def test_lut_graph_replay_matches_eager():
    t = torch()
    n, k = 5120, 17408
    w, _, _ = weights(TER, 370, n, k)
    x = dev(synth.gen_x(371, 1, k)[0])
    ws = sb.gemv_workspace(w)
    y0 = t.empty(n, dtype=t.float16, device="cuda")
    y1 = t.zeros(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv_ws(w, x, y0, ws)
    t.cuda.synchronize()
    s = t.cuda.Stream()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g, stream=s):
        for _ in range(3):
            sb.bonsai_gemv_ws(w, x, y1, ws)
    for _ in range(2):
        g.replay()
    t.cuda.synchronize()
    assert sb.bonsai_check_async() == 0
    assert counters(ws, n, k).max() == 0
    assert t.equal(y0.view(t.int16), y1.view(t.int16))


def test_lut_small_workspace_runs_streaming_kernel():
    """A workspace below the reported size runs bonsai_gemv's kernel (same
    bits) and leaves the buffer untouched."""
    t = torch()
    n, k = 17408, 5120
    w, _, _ = weights(TER, 380, n, k)
    x = dev(synth.gen_x(381, 1, k)[0])
    need = sb.bonsai_gemv_workspace_bytes(w)
    small = t.zeros(need - 256, dtype=t.uint8, device="cuda")
    y1 = t.empty(n, dtype=t.float16, device="cuda")
    y2 = t.empty(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv_ws(w, x, y1, small)
    sb.bonsai_gemv(w, x, y2)
    assert sb.bonsai_check_async() == 0
    assert t.equal(y1.view(t.int16), y2.view(t.int16))
    assert int(small.count_nonzero()) == 0


def test_lut_rejects_unaligned_workspace():
    t = torch()
    n, k = 17408, 5120
    w, _, _ = weights(TER, 382, n, k)
    x = dev(synth.gen_x(383, 1, k)[0])
    buf = t.zeros(sb.bonsai_gemv_workspace_bytes(w) + 512, dtype=t.uint8, device="cuda")
    y = t.empty(n, dtype=t.float16, device="cuda")
    with pytest.raises(sb.BonsaiError) as e:
        sb.bonsai_gemv_ws(w, x, y, buf[16:])
    assert "BONSAI_ERR_ALIGN" in str(e.value)


def test_lut_shapes_that_do_not_take_it():
    """K/128 not a multiple of 8 and too few rows per block report no
    workspace."""
    assert sb.bonsai_gemv_workspace_bytes(weights(BIN, 390, 4096, 5120)[0]) == 0
    assert sb.bonsai_gemv_workspace_bytes(weights(BIN, 395, 17408, 1280)[0]) == 0
    assert sb.bonsai_gemv_workspace_bytes(weights(BIN, 396, 17408, 5120)[0]) == 0
    assert sb.bonsai_gemv_workspace_bytes(weights(BIN, 397, 20000, 5120)[0]) > 0
    assert sb.bonsai_gemv_workspace_bytes(weights(TER, 391, 17408, 1280)[0]) == 0
    assert sb.bonsai_gemv_workspace_bytes(weights(TER, 392, 512, 5120)[0]) == 0
    assert sb.bonsai_gemv_workspace_bytes(weights(TER, 394, 4096, 5120)[0]) == 0
    assert sb.bonsai_gemv_workspace_bytes(weights(TER, 393, 17408, 5120)[0]) > 0
