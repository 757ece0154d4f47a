"""The entry point that allocates nothing, bonsai_gemv_splitk_static, against
bonsai_gemv and the oracle (needs a GPU).

It serves callers that may not allocate device memory while they run (a
decode loop that must not stall on cudaMalloc / cudaFree, or a process with a
fixed device-memory budget) and keeps its split-K partial sums in one fixed
device array instead. This file is collected last, so it runs both alone and
after every other GPU test of the session."""
import numpy as np
import pytest

import oracle
import sub_bit_weight_binary_b300 as sb
from sub_bit_weight_binary_b300 import synth
from gpu_util import TOL, assert_close, dev, host, torch, weights

pytestmark = pytest.mark.gpu
BIN, TER = sb.BONSAI_FMT_BINARY, sb.BONSAI_FMT_TERNARY


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch().cuda.is_available():
        pytest.skip("no CUDA device")
    sb.lib()


@pytest.mark.parametrize("fmt,n,k", [(BIN, 200, 17408), (TER, 77, 5120), (TER, 1000, 1280),
                                     (BIN, 8192, 1024), (TER, 16, 17408), (BIN, 1, 128)])
def test_no_alloc_matches_gemv(fmt, n, k):
    """Two consecutive calls give bit-identical y; both meet the oracle's bound
    and agree with bonsai_gemv to within the sum of the two bounds."""
    t = torch()
    w, packed, scales = weights(fmt, 80 + n % 13, n, k)
    x = synth.gen_x(81 + k % 7, 1, k)
    xd = dev(x[0])
    y0 = t.empty(n, dtype=t.float16, device="cuda")
    y1 = t.empty(n, dtype=t.float16, device="cuda")
    y2 = t.empty(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv(w, xd, y0)
    sb.bonsai_gemv_splitk_static(w, xd, y1)
    sb.bonsai_gemv_splitk_static(w, xd, y2)
    assert sb.bonsai_check_async() == 0
    assert t.equal(y1.view(t.int16), y2.view(t.int16))
    y_ref, nrm = oracle.linear(fmt, packed, scales, x)
    assert_close(host(y1), y_ref[0], nrm[0], "no-alloc fmt=%d n=%d k=%d" % (fmt, n, k))
    a = host(y0).view(np.float16).astype(np.float64)
    b = host(y1).view(np.float16).astype(np.float64)
    assert np.all(np.abs(a - b) <= 2 * TOL * nrm[0] + 1e-30)


def test_no_alloc_leaves_device_memory_untouched():
    """After a first call (the one-time set-up), a batch of calls changes the
    device's free memory by nothing: no allocation, by the library or by
    anything it calls."""
    t = torch()
    n, k = 640, 5120
    w, _, _ = weights(TER, 91, n, k)
    xd = dev(synth.gen_x(92, 1, k)[0])
    y = t.empty(n, dtype=t.float16, device="cuda")
    sb.bonsai_gemv_splitk_static(w, xd, y)
    t.cuda.synchronize()
    free0, _ = t.cuda.mem_get_info()
    for _ in range(50):
        sb.bonsai_gemv_splitk_static(w, xd, y)
    t.cuda.synchronize()
    free1, _ = t.cuda.mem_get_info()
    assert sb.bonsai_check_async() == 0
    assert free1 == free0


def test_no_alloc_rejects_more_rows_than_its_scratch():
    t = torch()
    n, k = 8193, 128
    w, _, _ = weights(BIN, 5, n, k)
    y = t.empty(n, dtype=t.float16, device="cuda")
    with pytest.raises(sb.BonsaiError) as e:
        sb.bonsai_gemv_splitk_static(w, dev(synth.gen_x(6, 1, k)[0]), y)
    assert "BONSAI_ERR_UNSUPPORTED" in str(e.value)
