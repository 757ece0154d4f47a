"""Decode plans (bonsai_decode_plan_init / bonsai_decode_run): many one-token
ternary products in one persistent launch, against the oracle (needs a GPU).

A plan computes the products of a decoder token in order inside one kernel;
a product whose x is an earlier product's y waits on that product's device
completion counter. Every step's output is compared with the oracle on the
inputs the step actually read."""
import numpy as np
import pytest

import oracle
import sub_bit_weight_binary_b300 as sb
from sub_bit_weight_binary_b300 import synth
from gpu_util import assert_close, assert_swiglu_close, dev, host, torch, weights

pytestmark = pytest.mark.gpu
TER = sb.BONSAI_FMT_TERNARY


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch().cuda.is_available():
        pytest.skip("no CUDA device")
    sb.lib()
    oracle.lib()
    yield
    assert sb.bonsai_check_async() == 0


def layer_plan(layers, hidden, ffn, seed):
    """Per layer: q||k||v and o read the layer's x; gate||up (SwiGLU) reads x
    and writes h; down reads h (after = the gate||up step)."""
    t = torch()
    steps, ref = [], []
    for layer in range(layers):
        x = synth.gen_x(seed + 100 * layer, 1, hidden)
        xd = dev(x[0])
        shapes = [("qkv", 3 * hidden, hidden), ("o", hidden, hidden),
                  ("gu", 2 * ffn, hidden), ("down", hidden, ffn)]
        h = t.empty(ffn, dtype=t.float16, device="cuda")
        for j, (name, n, k) in enumerate(shapes):
            w, packed, scales = weights(TER, seed + 10 * layer + j, n, k)
            if name == "gu":
                steps.append((w, xd, h, 1, -1))
                ref.append(("gu", packed, scales, x, h))
            elif name == "down":
                y = t.empty(n, dtype=t.float16, device="cuda")
                steps.append((w, h, y, 0, len(steps) - 1))
                ref.append(("down", packed, scales, h, y))
            else:
                y = t.empty(n, dtype=t.float16, device="cuda")
                steps.append((w, xd, y, 0, -1))
                ref.append((name, packed, scales, x, y))
    return steps, ref


def check_against_oracle(ref):
    for name, packed, scales, x, y in ref:
        if name == "gu":
            hh, g, u, ng, nu = oracle.swiglu(TER, packed, scales, x)
            assert_swiglu_close(host(y), hh[0], g[0], u[0], ng[0], nu[0], "plan gate/up")
        else:
            xin = host(x)[None, :] if name == "down" else x  # down read the GPU's h
            y_ref, nrm = oracle.linear(TER, packed, scales, xin)
            assert_close(host(y), y_ref[0], nrm[0], "plan %s" % name)


def test_plan_decoder_layers_match_oracle_and_repeat():
    steps, ref = layer_plan(3, 1280, 1024, 11)
    plan = sb.DecodePlan(steps)
    plan.run()
    assert sb.bonsai_check_async() == 0
    check_against_oracle(ref)
    first = [host(r[4]).copy() for r in ref]
    plan.run()  # the counters were reset by the first run
    plan.run()
    assert sb.bonsai_check_async() == 0
    for r, a in zip(ref, first):
        assert np.array_equal(host(r[4]), a)


def test_plan_dependent_chain():
    """y_j = W_j . y_{j-1}: every step waits for the one before it."""
    t = torch()
    k = 1280
    x0 = synth.gen_x(5, 1, k)
    xs = [dev(x0[0])]
    steps, mats = [], []
    for j in range(6):
        w, packed, scales = weights(TER, 40 + j, k, k)
        y = t.empty(k, dtype=t.float16, device="cuda")
        steps.append((w, xs[-1], y, 0, j - 1))
        mats.append((packed, scales))
        xs.append(y)
    plan = sb.DecodePlan(steps)
    plan.run()
    assert sb.bonsai_check_async() == 0
    for j, (packed, scales) in enumerate(mats):
        xin = host(xs[j])[None, :]
        y_ref, nrm = oracle.linear(TER, packed, scales, xin)
        assert_close(host(xs[j + 1]), y_ref[0], nrm[0], "chain step %d" % j)


def test_plan_in_cuda_graph_matches_eager():
    t = torch()
    steps, ref = layer_plan(2, 640, 512, 23)
    plan = sb.DecodePlan(steps)
    plan.run()
    assert sb.bonsai_check_async() == 0
    eager = [host(r[4]).copy() for r in ref]
    for r in ref:
        r[4].zero_()
    s = t.cuda.Stream()
    s.wait_stream(t.cuda.current_stream())
    g = t.cuda.CUDAGraph()
    with t.cuda.stream(s):
        with t.cuda.graph(g, stream=s):
            plan.run(stream=s)
    t.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    assert sb.bonsai_check_async() == 0
    for r, a in zip(ref, eager):
        assert np.array_equal(host(r[4]), a)


def test_plan_wait_that_never_arrives_times_out():
    """The dependency wait gives up after its limit and reports a timeout;
    the device stays usable and a plan runs correctly afterwards."""
    sb.bonsai_selftest_plan_wait(2_000_000)
    assert sb.STATUS[sb.bonsai_check_async()] == "BONSAI_ERR_TIMEOUT"
    assert sb.bonsai_check_async() == 0
    steps, ref = layer_plan(1, 640, 512, 31)
    plan = sb.DecodePlan(steps)
    plan.run()
    assert sb.bonsai_check_async() == 0
    check_against_oracle(ref)
